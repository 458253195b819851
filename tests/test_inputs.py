"""The seeded generators: deterministic, right shapes and distributions."""
import numpy as np
import torch

from comm_gemm_tile_gb300 import inputs as I


def test_deterministic_and_seed_sensitive():
    a1 = I.normal_bf16((64, 32), 1.0, 5)
    a2 = I.normal_bf16((64, 32), 1.0, 5)
    a3 = I.normal_bf16((64, 32), 1.0, 6)
    assert torch.equal(a1, a2) and not torch.equal(a1, a3)


def test_int_values_in_range():
    x = I.int_bf16((1000,), 1).float()
    assert set(torch.unique(x).tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_normal_std():
    x = I.normal_bf16((256, 256), 0.02, 3).float()
    assert abs(x.std().item() - 0.02) < 0.001


def test_zipf_popularity():
    lg = I.zipf_logits(20000, 64, 9)
    top1 = lg.argmax(1).numpy()
    share0 = np.mean(top1 == 0)
    p = np.arange(1, 65) ** -1.1
    assert abs(share0 - p[0] / p.sum()) < 0.02


def test_workload_shapes():
    w = I.AG_R8_TP8_UP
    assert (w.R, w.m, w.k, w.n) == (8, 1024, 8192, 3584)
    assert abs(w.flops() - 4.81e11) / 4.81e11 < 0.01
    w = I.RS_R8_TP8_DOWN
    assert abs(w.flops() - 3.85e12) / 3.85e12 < 0.01
    a, b = I.gemm_inputs(I.RS_R2_256_INT)
    assert len(a) == 2 and a[0].shape == (256, 256) and b[1].shape == (256, 256)


def test_sample_rows_cover_tiles():
    rows = I.sample_rows(1000, 0)
    assert rows[0] == 0 and rows[-1] == 999
    assert set(range(0, 1000, 128)) <= set((r // 128) * 128 for r in rows)
