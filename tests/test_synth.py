"""The seeded input generator: storage rounding, row addressing and the workload recipe."""
import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(size=10000), rng.normal(size=1000) * 1e-30,
                        [0.0, -0.0, 1.0, 1.00390625, 1.0 + 2 ** -9, 1.0 + 3 * 2 ** -9, 65504.0]])
    x = x.astype(np.float32)
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_rows_are_addressable():
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=12, seqlen=33)
    full = synth.scan_inputs(cfg)
    rows = [23, 0, 5, 12]
    sub = synth.scan_rows(cfg, rows)
    for k in ("u", "delta", "z"):
        assert np.array_equal(sub[k], full[k].reshape(-1, 33)[rows])
    # a longer sequence starts with the same values (row streams do not depend on L's use)
    again = synth.scan_inputs(cfg)
    assert all(np.array_equal(again[k], full[k]) for k in ("u", "delta", "z", "B", "C"))


def test_recipe_delta_range_and_params():
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=64, seqlen=512)
    inp = synth.scan_inputs(cfg)
    dt = np.logaddexp(0.0, inp["delta"].astype(np.float64) + inp["delta_bias"][None, :, None])
    assert dt.min() >= synth.DELTA_MIN * (1 - 1e-5) and dt.max() <= synth.DELTA_MAX * (1 + 1e-5)
    assert np.array_equal(inp["A"][3], -np.arange(1, 17, dtype=np.float32))
    assert abs(inp["u"].std() - 1.0) < 0.05 and abs(inp["D"].mean() - 1.0) < 0.05
    tiny = synth.scan_inputs(synth.CONFIGS["tiny"])
    assert np.all(tiny["D"] == 1.0) and np.all(tiny["delta_bias"] == 0.0)
    assert tiny["B"].shape == (1, 4, 64)


def test_bf16_workload_is_rounded_fp32():
    cfg = synth.CONFIGS["b14"].replace(batch=1, dim=4, seqlen=16)
    a = synth.scan_inputs(cfg)
    b = synth.scan_inputs(cfg.replace(dtype="f32"))
    for k in ("u", "z", "B", "C", "delta"):
        assert a[k].dtype == np.uint16
        assert np.array_equal(a[k], synth.f32_to_bf16_bits(b[k]))


def test_decode_inputs_subset():
    cfg = synth.CONFIGS["decode"].replace(batch=3, dim=8, decode_steps=4)
    allin = synth.decode_inputs(cfg)
    one = synth.decode_step_inputs(cfg, 2, batches=[1])
    for k in ("x", "delta", "z", "B", "C"):
        assert np.array_equal(one[k][0], allin[k][2, 1])
    h = synth.decode_state0(cfg)
    assert h.shape == (3, 8, 16) and np.array_equal(synth.decode_state0(cfg, [2])[0], h[2])


def test_backward_inputs_are_addressable_and_seeded():
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=6, dstate=5, seqlen=21)
    g = synth.grad_inputs(cfg)
    assert g["dy"].shape == (2, 6, 21) and g["dlast"].shape == (2, 6, 5) and g["h0"].shape == (2, 6, 5)
    rows = [11, 0, 7]
    assert np.array_equal(synth.grad_rows(cfg, rows), g["dy"].reshape(-1, 21)[rows])
    assert np.array_equal(synth.state_rows(cfg, rows, "h0"), g["h0"].reshape(-1, 5)[rows])
    # the gradient streams differ from the input streams and from each other
    inp = synth.scan_inputs(cfg)
    assert not np.array_equal(g["dy"], inp["u"]) and not np.array_equal(g["h0"], g["dlast"])
    bf = synth.grad_inputs(cfg.replace(dtype="bf16"))
    assert bf["dy"].dtype == np.uint16 and np.array_equal(bf["dy"], synth.f32_to_bf16_bits(g["dy"]))


def test_convolution_recipe():
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=300, seqlen=8)
    for K in (1, 2, 4):
        p = synth.conv_params(cfg, K)
        lim = 1.0 / np.sqrt(K)
        assert p["conv_w"].shape == (300, K) and p["conv_bias"].shape == (300,)
        assert np.all(np.abs(p["conv_w"]) <= lim) and np.all(np.abs(p["conv_bias"]) <= lim)
        assert abs(float(np.mean(p["conv_w"]))) < 0.1 * lim
        assert np.array_equal(synth.conv_params(cfg, K)["conv_w"], p["conv_w"])  # seeded
        assert synth.conv_prev(cfg, K).shape == (2, 300, K - 1)
