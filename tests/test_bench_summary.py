"""The bench line's compact per-row summary (host logic, no GPU): every row
the bench measures appears with its value, its fraction of the bound and the
same-run vendor-library figure, in few enough characters that the end of
the bench's stdout always holds all of it."""
import json

import bench

PEAKS = {"bf16_tflops": 1900.4, "hbm_gbs": 6782.4, "bf16_tflops_sustained": 1704.5}


def fake_rows():
    sk = {}
    for key in ("128x8192x16384", "4096x4096x512", "1000x1000x1000"):
        sk[key] = {"us": 20.0, "tflops": 700.0, "roofline_tflops": 1900.4, "frac": 0.37, "grid": 148,
                   "role_timeline": {"producer_wait_empty_share": 0.1},
                   "splitk": {"us": 30.0, "tflops": 650.0, "frac": 0.3, "splits": 2, "grid": 148, "atom": 1,
                              "tile_n": 128},
                   "cpu_oracle": {"sample": "full", "macs": 1, "seconds": 1.0}}
    lib = {"conv_32x56x56x256_3x3": {"us": 70.3, "tflops": 1684.6},
           "gemm_8192x8192x8192": {"us": 551.5, "tflops": 1993.5},
           "gemm_320x200x448": {"us": 6.8, "tflops": 8.5},
           "copy_1GiB": {"gbs": 6764.7}, "transpose_1GiB": {"gbs": 1092.1}}
    for key in sk:
        lib[f"gemm_{key}"] = {"us": 19.0, "tflops": 900.0}
    return {
        "conv_32x56x56x256_3x3": {"unit": "TFLOP/s", "auto": {"us": 72.3, "tflops": 1637.0, "frac_of_peak": 0.861,
                                                             "atom": 2, "tile_n": 256, "pipe_depth": 6}},
        "skinny_gemm_set": {"unit": "TFLOP/s", "l2": "flushed between calls", **sk},
        "gemm_320x200x448_f32": {"unit": "us", "mean_us": 10.9, "min_us": 8.8},
        "tma_copy_1GiB": {"gbs": 6790.5, "frac_of_hbm": 1.001, "bit_exact": True},
        "tma_transpose_1GiB": {"gbs": 6556.1, "frac_of_hbm": 0.967, "bit_exact": True},
        "fallback_paths": {"plain_load_producer_4096": {"tflops": 28.1},
                           "tma_producer_4096_same_variant": {"tflops": 1446.6}},
        "library_comparison": lib,
    }


def fake_sweep():
    out = []
    for atom, tile_n, depths in ((1, 64, range(2, 10)), (1, 128, range(2, 8)), (2, 128, range(2, 10)),
                                 (1, 256, range(2, 6)), (2, 256, range(2, 8))):
        for d in depths:
            out.append({"atom": atom, "tile_n": tile_n, "pipe_depth": d, "tflops": 1234.5})
    return out


def test_summary_names_every_row_with_its_bound_and_library_figure():
    s = bench.summarize(2005.6, 2005.6, 1900.4, fake_rows(), fake_sweep(), PEAKS)
    for key in ("gemm_8192x8192x8192", "conv_32x56x56x256_3x3", "gemm_128x8192x16384", "gemm_4096x4096x512",
                "gemm_1000x1000x1000", "gemm_320x200x448_f32", "tma_copy_1GiB", "tma_transpose_1GiB",
                "depth_sweep_tflops"):
        assert key in s, key
    assert s["conv_32x56x56x256_3x3"]["cudnn_tflops"] == 1684.6
    assert s["gemm_4096x4096x512"]["cublas_tflops"] == 900.0
    assert s["gemm_8192x8192x8192"]["frac"] == round(2005.6 / 1900.4, 3)
    assert len(s["depth_sweep_tflops"]["2/256"]) == 6
    assert len(json.dumps(s)) < 2500


def test_summary_without_rows_keeps_the_headline():
    s = bench.summarize(1700.0, 1700.0, 1704.5, None, None, PEAKS)
    assert set(s) == {"gemm_8192x8192x8192", "peaks"}
