"""CPU oracle for the OIDN-style U-Net denoiser forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the package
`conv2d_implicit_gemm_gb300`, its C-ABI library or its kernels) imports,
links or runs this code.  Only `tests/`, `__graft_entry__.smoke()` and the
`cpu_baseline` / `--impl reference` legs of `bench.py` may use it.

It is a plain, slow restatement of what the pages define, in numpy float64:

* `numerics`  - fp16/fp32 storage rounding, sanitize, the HDR transfer pair;
* `layers`    - same-padded 3x3 conv + bias (+ReLU), 2x2 max-pool,
                nearest 2x upsample, channel concat;
* `passes`    - the per-tile input pass (pack) and output pass (unpack);
* `tiles`     - the overlapping tile grid and the network's dependency radius;
* `unet`      - the 16-layer network and the whole tiled denoise.

Sources (web pages, cited by title and function/section):

* "oidn-web 0.3.4 -> 0.4.0, package/src/nativeUNet.ts" (conv, pool,
  decoder, input-pack shaders; weight packer; activation plan);
* "oidn-web 0.4.0 -> 0.5.0, package/src/nativeUNet.ts" (implicit-GEMM
  tuning, decoder variants);
* "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts" (input pass,
  output pass, tile grid use).

Where the pages are silent, ambiguous or garbled, the oracle takes a
reading of them; each function states the reading it uses in its own
docstring.

Parity status: every function here is pinned by `tests/test_oracle_*.py`
against library routines (torch CPU float64 conv2d / max_pool2d /
interpolate), closed forms, invariants or brute force; none is unpinned.
"""
