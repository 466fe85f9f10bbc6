"""The lookup tables compiled into the CUDA library are exactly what their
committed generators produce (no stale or hand-edited table).  CPU only."""
import io
import os
import runpy

import pytest

KERN = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "modulation_bit_exact_gb300", "csrc", "kernels")


@pytest.mark.parametrize("gen,inc", [("gen_tanh_table.py", "tanh_bf16_table.inc"),
                                     ("gen_rstd_table.py", "rstd_bf16_table.inc")])
def test_generated_table_is_current(gen, inc):
    mod = runpy.run_path(os.path.join(KERN, gen))
    buf = io.StringIO()
    mod["main"](buf)
    with open(os.path.join(KERN, inc)) as f:
        assert f.read() == buf.getvalue()
