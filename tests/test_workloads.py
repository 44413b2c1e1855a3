"""The seeded input recipes: shapes, dtypes, mask fractions and determinism."""
import torch

import workloads as wl


def test_five_workloads_and_flops():
    names = [w.name for w in wl.WORKLOADS]
    assert names == ["tiny", "qwen2_7b", "qwen3_8b", "long_ctx", "stress"]
    q2 = wl.get("qwen2_7b")
    assert (q2.N, q2.H, q2.V) == (8192, 3584, 152064)
    assert q2.flops == 8 * 8192 * 3584 * 152064


def test_label_masks_full_N_small_vocab():
    # full token counts and mask recipes; H and V cut down to keep this fast
    for w in wl.WORKLOADS:
        X, W, lab = wl.make_inputs(w, H=16, V=min(w.V, 4096) if w.labels != "zipf" else w.V)
        assert X.dtype == torch.bfloat16 and W.dtype == torch.bfloat16
        assert lab.dtype == torch.int64 and lab.shape == (w.N,)
        frac = (lab == -100).float().mean().item()
        assert abs(frac - w.mask_frac) < 0.01, (w.name, frac)
        ok = lab[lab != -100]
        assert ok.min() >= 0 and ok.max() < W.shape[0]
    lc = wl.make_inputs(wl.get("long_ctx"), H=8, V=64)[2]
    assert (lc[:13107] == -100).all() and (lc[13107:] != -100).all()
    q3 = wl.make_inputs(wl.get("qwen3_8b"), H=8)[2].view(2, 4, 2048)
    assert (q3[:, :, :410] == -100).all() and (q3[:, :, 410:] != -100).all()


def test_zipf_prefers_low_ids():
    lab = wl.make_inputs(wl.get("qwen3_8b"), H=8)[2]
    lab = lab[lab != -100]
    assert (lab < 100).float().mean() > 0.3


def test_rms_rows_and_determinism():
    w = wl.get("qwen3_8b")
    X, _, _ = wl.make_inputs(w, N=64, H=256, V=32)
    rms = X.float().pow(2).mean(1).sqrt()
    assert torch.allclose(rms, torch.ones_like(rms), atol=1e-2)
    a = wl.make_inputs(wl.get("tiny"))
    b = wl.make_inputs(wl.get("tiny"))
    assert all(torch.equal(x, y) for x, y in zip(a, b))
