"""The oracle: a plain, slow, obviously correct CPU restatement of the fused
grouped-MLP forward with MXFP8 / NVFP4 block quantisation and of the group
quantisers.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
bench.py's CPU-baseline leg may import it.  It shares no code with the CUDA
path (``mxfp8_nvfp4_block_gb300``) and never imports it; the two meet only in
the seeded input generators, which hold none of the method's arithmetic.

Layout:
  formats.c  -- E4M3 / E2M1 / E8M0 / bf16 rounding, MXFP8 and NVFP4 block
                quantisation, the 16-point RHT, group (Hadamard-)amax,
                columnwise NVFP4 (C, compiled by ``build()``)
  quant.py   -- group quantisers (``group_quantize``, ``group_hadamard_amax``,
                ``group_quantize_with_amax``)
  forward.py -- the forward (``forward``) and per-expert weight quantisation
  backward.py -- the backward's data gradients (``backward_dgrad``) and weight
                gradients (``backward_wgrad``, columnwise MXFP8 ``mxfp8_colwise``)
  layout.py  -- the boundary's scale layouts (COMPACT, GEMM_TILED)

Parity pins live in tests/test_oracle_*.py.  Functions without a pin: none.
"""
from ._lib import build, lib  # noqa: F401
from .backward import (backward_dgrad, backward_wgrad, dact, mxfp8_colwise, padded_offsets,  # noqa: F401
                       recompute_fc2x)
from .forward import SRELU, SWIGLU, TANH_SRELU, activation, dequant_weight, forward, quantize_weights  # noqa: F401
from .layout import (compact_to_tiled, group_offsets, tile_bases, tiled_index, tiled_size,  # noqa: F401
                     tiled_to_compact, tiled_to_x4)
from .quant import (MXFP8, NVFP4, amax_bf16, bf16_to_f64, f64_to_bf16, group_amax,  # noqa: F401
                    group_hadamard_amax, group_quantize, group_quantize_with_amax, mxfp8_dequant_rows,
                    mxfp8_quantize_rows, nvfp4_dequant_rows, nvfp4_global_scale, nvfp4_quantize_block,
                    nvfp4_quantize_rows, rht16)
