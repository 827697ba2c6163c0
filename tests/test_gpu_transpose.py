"""GPU checks of the TMA transpose (and its fallback): bit-exact against the
source's transpose, destination pitch padding untouched, every ring shape,
ragged edges, misaligned buffers and the full 1 GiB workload."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen  # noqa: E402
import mbarrier_pipelined_tensor_gb300 as tp  # noqa: E402
from gpu_util import dev_u16, expect_ok, host_u16  # noqa: E402

pytestmark = pytest.mark.gpu
MARK = 0x2D2D


def run_transpose(rows, cols, ld_src, ld_dst, seed, **opts):
    src_h = datagen.copy_source(rows, cols, seed=seed, ld=ld_src)
    src = dev_u16(src_h)
    dst = torch.full((cols, ld_dst), MARK, dtype=torch.int16, device="cuda")
    if opts:
        tp.tp_tma_transpose_2d_ex(src, dst, rows, cols, ld_src, ld_dst, **opts)
    else:
        tp.tp_tma_transpose_2d(src, dst, rows, cols, ld_src, ld_dst)
    expect_ok()
    got = host_u16(dst)
    assert np.array_equal(got[:, :rows], src_h[:, :cols].T)
    assert np.all(got[:, rows:] == MARK), "wrote into the destination pitch padding"
    return tp.tp_last_plan()


@pytest.mark.parametrize("rows,cols,ld_src,ld_dst", [(256, 512, 512, 256), (300, 1000, 1000, 304),
                                                     (1000, 130, 136, 1008), (777, 1500, 1504, 784),
                                                     (64, 4096, 4096, 72)])
def test_tma_transpose_bit_exact(rows, cols, ld_src, ld_dst):
    plan = run_transpose(rows, cols, ld_src, ld_dst, seed=rows + cols)
    assert plan["path"] == tp.TP_PATH_TMA_TRANSPOSE


@pytest.mark.parametrize("stages,per_sm", [(2, 1), (4, 4), (6, 2), (8, 3)])
def test_tma_transpose_ring_shapes(stages, per_sm):
    plan = run_transpose(1030, 2050, 2056, 1032, seed=9, stages=stages, ctas_per_sm=per_sm)
    assert plan["path"] == tp.TP_PATH_TMA_TRANSPOSE and plan["pipe_depth"] == stages


@pytest.mark.parametrize("rows,cols,ld_src,ld_dst", [(100, 1001, 1001, 100), (33, 17, 19, 40), (500, 600, 600, 500),
                                                     (129, 67, 70, 131), (64, 64, 65, 65), (1, 300, 300, 1),
                                                     (300, 1, 1, 301)])
def test_transpose_fallback(rows, cols, ld_src, ld_dst):
    plan = run_transpose(rows, cols, ld_src, ld_dst, seed=3)
    assert plan["path"] == tp.TP_PATH_VEC_TRANSPOSE or (rows * cols * 2 >= 65536 and plan["path"] ==
                                                        tp.TP_PATH_TMA_TRANSPOSE)
    plan = run_transpose(rows, cols, ld_src, ld_dst, seed=3, force_vec=True)
    assert plan["path"] == tp.TP_PATH_VEC_TRANSPOSE


def test_transpose_misaligned_base():
    rows, cols = 300, 400
    total = rows * cols + 8
    src_h = datagen.Stream(12).bits16((total,))
    src_all = dev_u16(src_h)
    dst_all = torch.full((cols * rows + 8,), MARK, dtype=torch.int16, device="cuda")
    tp.tp_tma_transpose_2d(src_all[1:], dst_all[3:], rows, cols, cols, rows)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_VEC_TRANSPOSE
    got = host_u16(dst_all)
    want = src_h[1:1 + rows * cols].reshape(rows, cols).T.reshape(-1)
    assert np.array_equal(got[3:3 + rows * cols], want)
    assert np.all(got[:3] == MARK) and np.all(got[3 + rows * cols:] == MARK)


def test_transpose_1gib_bit_exact():
    rows, cols = 32768, 16384
    src = dev_u16(datagen.copy_source(rows, cols, seed=4))
    dst = torch.empty((cols, rows), dtype=torch.int16, device="cuda")
    tp.tp_tma_transpose_2d(src, dst, rows, cols, cols, rows)
    expect_ok()
    assert tp.tp_last_plan()["path"] == tp.TP_PATH_TMA_TRANSPOSE
    assert torch.equal(dst, src.t())
