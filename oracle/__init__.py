"""Float64 CPU oracle for chunked Gated DeltaNet prefill — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import, call or execute anything
in this package.  The product path (the CUDA library and its binding) never
touches it, and this package imports nothing from the product package.

Contents
--------
``token_loop``  the plain definition: the gated delta rule one token at a time
                in float64 (C, compiled from ``gdn_oracle.c``), with the
                optional short convolution and q/k L2 normalisation in front.
``chunk_form``  the chunked closed form of the Qwen3.5 chunked-prefill pull
                request ("perf(qwen3_5): prefill text prompts in multi-token
                chunks", Implementation), in float64 NumPy, with the two
                triangular inverses (forward substitution and the blocked
                8x8-Neumann / 2x2-level scheme).  It is used to pin the token
                loop, not as a second reference for the GPU.
``scan_rows``   the selective-scan rows of the Mamba chunked-prefill pull
                request (h_t = a_t h_{t-1} + b_t): the plain row loop (C) and
                the page's chunked Hillis-Steele doubling scan (NumPy).
``wkv_rows``    the RWKV-4 WKV of the RWKV chunked-prefill pull request: the
                decoder's (num, den, max) recurrence row by row (C) and the
                page's chunk form with per-row max shift (NumPy).
``attn_rows``   full-attention rows over a KV cache plus the chunk's causal
                prefix (the Qwen3.5 page's full-attention layers), float64
                NumPy.
"""

from .token_loop import (build_oracle, oracle_prefill, oracle_step, oracle_short_conv,  # noqa: F401
                         oracle_l2norm, max_threads)
from . import chunk_form  # noqa: F401
from . import scan_rows  # noqa: F401
from . import wkv_rows  # noqa: F401
from . import attn_rows  # noqa: F401
