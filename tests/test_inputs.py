"""The seeded generator: determinism, shapes and the workload statistics it promises."""
import numpy as np
import torch

from latent_moe_layer_route_gb300 import configs, inputs
from oracle import model as T


def test_deterministic_and_shapes():
    cfg = configs.SMALL
    a1, w1 = inputs.make_inputs(cfg)
    a2, w2 = inputs.make_inputs(cfg)
    for k in a1:
        assert torch.equal(a1[k], a2[k])
    for k in w1:
        assert torch.equal(w1[k], w2[k])
    assert a1["x"].shape == (cfg.M, cfg.H) and a1["x"].dtype == torch.bfloat16
    assert a1["z"].shape == (cfg.M, cfg.L) and a1["z"].dtype == torch.bfloat16
    assert a1["logits"].shape == (cfg.M, cfg.E) and a1["logits"].dtype == torch.float32
    assert w1["w13_q"].shape == (cfg.E, 2 * cfg.I, cfg.L)
    assert w1["w13_s"].shape == (cfg.E, 2 * cfg.I // 128, cfg.L // 128)
    assert w1["w2_q"].shape == (cfg.E, cfg.L, cfg.I)
    assert w1["ws13"].shape == (2 * cfg.Is, cfg.H)
    assert w1["ws2"].shape == (cfg.H, cfg.Is)
    assert w1["w_up"].shape == (cfg.H, cfg.L)


def test_activation_prefix_is_stable_in_m():
    # weights do not depend on M; a smaller M draws from the same stream
    cfg = configs.SMALL
    w_a = inputs.make_weights(cfg.with_(M=3))
    w_b = inputs.make_weights(cfg.with_(M=50))
    assert torch.equal(w_a["w13_q"], w_b["w13_q"])


def test_fp8_block_quantize_error_bound():
    g = torch.Generator().manual_seed(0)
    w = torch.randn(256, 384, generator=g) * 0.05
    q, s = inputs.fp8_block_quantize(w)
    d = T.dequant_fp8_blocks(q.numpy(), s.numpy())
    err = np.abs(d - w.double().numpy())
    bound = np.abs(w.double().numpy()) / 16 + np.repeat(np.repeat(s.numpy(), 128, 0), 128,
                                                        1) * 2.0 ** -10
    assert (err <= bound * (1 + 1e-6)).all()


def test_nvfp4_quantize_error_bound():
    g = torch.Generator().manual_seed(1)
    w = torch.randn(64, 256, generator=g) * 0.03
    packed, sb, gs = inputs.nvfp4_quantize(w)
    d = T.dequant_nvfp4(packed.numpy(), sb.numpy(), gs)
    # error within half an e2m1 step of the block scale plus the e4m3 scale rounding
    blk = np.abs(w.numpy()).reshape(64, 16, 16).max(-1)
    err = np.abs(d - w.double().numpy()).reshape(64, 16, 16).max(-1)
    assert (err <= blk * 0.25 + 1e-9).all()


def test_zipf_skew_and_bias_recipes():
    c3 = configs.PREFILL_M4096
    act = inputs.make_activations(c3)
    load = inputs.expert_load(act["logits"], c3.topk)
    assert load.sum() == c3.M * c3.topk
    assert load.max() > 3 * load.mean()
    assert load.argmax() == 0
    c2 = configs.DECODE_M128
    load2 = inputs.expert_load(inputs.make_activations(c2)["logits"], c2.topk)
    assert load2.max() > 2 * load2.mean()
