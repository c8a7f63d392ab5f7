"""CPU oracle for exact softmax attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the library (``paged_kv_decode_17_gb300``)
imports, links or runs this package; only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code, tables or helpers with the CUDA path; both sides receive their
inputs from ``workloads`` (random numbers and page assignments only).

Everything is plain numpy in float64 (or pure Python in ``brute``), one
(sequence, head) at a time, with the whole score row materialised: the plain
definition of attention that the tiled/split kernels must reproduce.

Modules
-------
``attention``  materialised-score attention over gathered pages, and the
               K/V writeback scatter (the reference definitions).
``brute``      an independent scalar pure-Python restatement, for tiny inputs.
``fp8``        the e4m3 code table, the quantising FP8 writeback and attention
               over dequantised FP8 pages.
``rope``       the rotary position embedding and RMS normalisation that the
               fused writeback applies to K (and Q) rows, and bf16 rounding.
``tiled``      a CPU model of the online-softmax recurrence and of the
               log-sum-exp combine of split chunks, used to pin that the
               tiled/split algorithm equals the materialised one.

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""

from .attention import (  # noqa: F401
    bf16_bits_to_f64,
    gather_kv_rows,
    attention_rows,
    paged_attention,
    kv_write_paged,
)
from .fp8 import (  # noqa: F401
    e4m3_decode,
    e4m3_encode,
    kv_write_paged_fp8,
    paged_attention_fp8,
)
from .rope import (  # noqa: F401
    bf16_ulp,
    rms_norm,
    rope_angles,
    rope_rotate_half,
    rope_writeback_rows,
    round_to_bf16_f64,
)
