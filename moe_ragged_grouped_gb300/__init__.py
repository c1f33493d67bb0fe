"""GB300 (sm_103a) ragged BF16 grouped GEMM: forward, data gradient, weight gradient.

The compute path is the C-ABI library ``libcake_gg.so`` (hand-written CUDA for
sm_103a: TMA, tcgen05 MMAs into TMEM, persistent ragged tile walk).  The
Python module ``cake_gg`` is a ctypes binding with the same names as the C
entry points; ``workloads`` draws seeded synthetic inputs.
"""
from . import cake_gg, workloads  # noqa: F401
from .cake_gg import (  # noqa: F401
    cake_gg_check_status, cake_gg_dgrad, cake_gg_fwd, cake_gg_plan, cake_gg_strerror,
    cake_gg_tile_walk, cake_gg_wgrad, grouped_gemm,
)
