"""The TMA read stream (tp_tma_read_2d): the load half of the copy ring on
its own, used as the measured bound of a GEMM that streams its B once. It
must complete on every tile shape and ring depth it accepts, including a
ragged last tile row and column, leave its source untouched, and refuse
buffers TMA cannot describe."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import dev_u16, expect_ok, host_u16  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,ld", [(1000, 1000, 1000), (4096, 2048, 2048), (333, 72, 80)])
@pytest.mark.parametrize("opts", [dict(), dict(stages=2), dict(stages=12, box_rows=64), dict(box_rows=256, stages=4),
                                  dict(ctas_per_sm=2, stages=4)])
def test_read_stream_runs_and_leaves_source(rows, cols, ld, opts):
    src = datagen.copy_source(rows, ld, seed=31)
    s = dev_u16(src)
    tp.tp_tma_read_2d(s, rows, cols, ld, **opts)
    expect_ok()
    plan = tp.tp_last_plan()
    assert plan["path"] == tp.TP_PATH_TMA_READ and plan["grid"] >= 1
    assert plan["pipe_depth"] == opts.get("stages", 8)
    assert np.array_equal(host_u16(s), src)


def test_read_stream_refuses_what_tma_cannot_describe():
    s = torch.zeros(4096 * 4, dtype=torch.int16, device="cuda")
    for args in ((s[1:], 64, 64, 64), (s, 64, 60, 64), (s, 64, 64, 68)):
        with pytest.raises(tp.TPError) as e:
            tp.tp_tma_read_2d(*args)
        assert e.value.status == tp.TP_ERR_UNSUPPORTED
    with pytest.raises(tp.TPError) as e:
        tp.tp_tma_read_2d(s, 64, 64, 64, stages=3)
    assert e.value.status == tp.TP_ERR_INVALID_ARG
