"""Pins of the float64 oracle to things other than itself: library routines that compute
the same step by another route, closed forms, invariants, special cases and a scalar
brute-force re-derivation on tiny shapes."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import brute
from latent_moe_layer_route_gb300 import configs, inputs
from oracle import model as T
from oracle.codecs import e4m3_decode


# ------------------------------------------------------------------ routing

def test_route_matches_torch_topk_and_softmax():
    rng = np.random.default_rng(0)
    lg = rng.standard_normal((64, 32)).astype(np.float32)
    ids, w = T.route(lg, 6)
    tv, ti = torch.topk(torch.from_numpy(lg).double(), 6, dim=1)
    assert np.array_equal(ids, ti.numpy())
    ref = torch.softmax(tv, dim=1).numpy()
    np.testing.assert_allclose(w, ref, rtol=1e-14, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)


def test_route_ties_prefer_lower_index_and_weights_equal():
    lg = np.zeros((2, 8), dtype=np.float32)
    lg[1, [2, 5, 6]] = 3.0
    ids, w = T.route(lg, 3)
    assert ids[0].tolist() == [0, 1, 2]
    assert ids[1].tolist() == [2, 5, 6]
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-15)


def test_route_shift_invariance():
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((16, 16)).astype(np.float32)
    i1, w1 = T.route(lg, 4)
    i2, w2 = T.route(lg + np.float32(8.0), 4)
    assert np.array_equal(i1, i2)
    np.testing.assert_allclose(w1, w2, rtol=1e-5)


# ------------------------------------------------------------------ permutation

def test_permutation_matches_loops():
    rng = np.random.default_rng(2)
    M, E, k = 37, 9, 3
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    cnt, off, gidx, slot, pos = T.permutation(ids, E)
    lists = [[] for _ in range(E)]
    for t in range(M):
        for j in range(k):
            lists[ids[t, j]].append((t, j))
    flat = [tj for e in range(E) for tj in lists[e]]
    assert cnt.tolist() == [len(x) for x in lists]
    assert off.tolist() == [0] + list(np.cumsum([len(x) for x in lists]))
    assert gidx.tolist() == [t for t, _ in flat]
    assert slot.tolist() == [t * k + j for t, j in flat]
    for p, (t, j) in enumerate(flat):
        assert pos[t, j] == p


def test_permutation_is_inverse_of_pos():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((50, 12)).astype(np.float32)
    ids, _ = T.route(lg, 4)
    cnt, off, gidx, slot, pos = T.permutation(ids, 12)
    k = 4
    for t in range(50):
        for j in range(k):
            p = pos[t, j]
            assert slot[p] == t * k + j and gidx[p] == t
            assert off[ids[t, j]] <= p < off[ids[t, j] + 1]


# ------------------------------------------------------------------ activation quant

def test_quant_per128_matches_scalar_rule():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal((3, 256)) * rng.uniform(0.01, 30, (3, 1))).astype(np.float32)
    v[2, 128:] = 0.0  # an all-zero group takes scale 1 and zero codes
    q, s = T.quant_per128(v)
    for i in range(3):
        for g in range(2):
            bq, bs = brute.quant_group([float(x) for x in v[i, g * 128:(g + 1) * 128]])
            assert q[i, g * 128:(g + 1) * 128].tolist() == bq
            assert float(s[i, g]) == bs
    assert s[2, 1] == 1.0 and not q[2, 128:].any()


def test_quant_per128_error_bound_and_amax_code():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 512)).astype(np.float32)
    q, s = T.quant_per128(v)
    deq = e4m3_decode(q).reshape(64, 4, 128) * s[..., None]
    err = np.abs(deq.reshape(64, 512) - v)
    # e4m3 has 3 mantissa bits: relative half-step 1/16 in the normal range, plus the
    # subnormal absolute half-step 2^-10 * s.
    bound = np.abs(v) / 16 + np.repeat(s, 128, axis=1) * 2.0 ** -10
    assert (err <= bound * (1 + 1e-6)).all()
    # the element holding the group amax maps to the largest code, 448
    a = np.abs(v.reshape(64, 4, 128)).argmax(-1)
    qq = q.reshape(64, 4, 128)
    top = np.take_along_axis(qq, a[..., None], -1)[..., 0] & 0x7F
    assert (top == 0x7E).all()


# ------------------------------------------------------------------ pieces vs library

def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(6)
    r = rng.standard_normal((8, 384)) * 3.0
    g = rng.uniform(0.5, 1.5, 384)
    ours = T.rmsnorm(r, g, 1e-6)
    ref = F.rms_norm(torch.from_numpy(r), (384,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(ours, ref, rtol=1e-13, atol=1e-13)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(7)
    r = rng.standard_normal((4, 256))
    n = T.rmsnorm(r, np.ones(256), 0.0)
    np.testing.assert_allclose(np.sqrt((n * n).mean(1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(T.rmsnorm(37.5 * r, np.ones(256), 0.0), n, rtol=1e-12)


def test_swiglu_mlp_matches_torch_functional():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, 96))
    w13 = rng.standard_normal((2 * 40, 96))
    w2 = rng.standard_normal((72, 40))
    xt, w13t, w2t = map(torch.from_numpy, (x, w13, w2))
    h = F.linear(xt, w13t)
    ref = F.linear(F.silu(h[:, :40]) * h[:, 40:], w2t).numpy()
    np.testing.assert_allclose(T.swiglu_mlp(x, w13, w2), ref, rtol=1e-12, atol=1e-12)
    assert T.silu(np.array([0.0]))[0] == 0.0


def test_dequant_fp8_blocks_matches_loops():
    rng = np.random.default_rng(9)
    q = rng.integers(0, 0x7E, (256, 384)).astype(np.uint8)
    s = rng.uniform(0.001, 1.0, (2, 3)).astype(np.float32)
    d = T.dequant_fp8_blocks(q, s)
    for (i, j) in [(0, 0), (127, 128), (128, 383), (255, 200), (77, 260)]:
        assert d[i, j] == e4m3_decode(q[i:i + 1, j:j + 1])[0, 0] * float(s[i // 128, j // 128])


def test_dequant_nvfp4_matches_loops():
    rng = np.random.default_rng(10)
    R, C = 4, 64
    packed = rng.integers(0, 256, (R, C // 2)).astype(np.uint8)
    sb = rng.integers(0, 0x7E, (R, C // 16)).astype(np.uint8)
    g = 0.37
    d = T.dequant_nvfp4(packed, sb, g)
    for i in range(R):
        for k in range(C):
            byte = int(packed[i, k // 2])
            code = byte & 0xF if k % 2 == 0 else byte >> 4
            ref = brute.e2m1_value(code) * (brute.e4m3_value(int(sb[i, k // 16])) * g)
            assert d[i, k] == ref


def test_generator_nvfp4_roundtrip_of_representable_weights():
    # Weights built from e2m1 values times an exact block scale come back unchanged.
    rng = np.random.default_rng(11)
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)
    w = rng.choice(vals, (8, 64)) * rng.choice([-1, 1], (8, 64))
    w[:, ::16] = 6.0  # every block reaches the max code so the block scale is exact
    w = torch.from_numpy((w * 0.25).astype(np.float32))
    packed, sb, g = inputs.nvfp4_quantize(w)
    np.testing.assert_allclose(T.dequant_nvfp4(packed.numpy(), sb.numpy(), g), w.numpy(),
                               rtol=1e-6, atol=0)


# ------------------------------------------------------------------ special cases

def _small(**kw):
    cfg = configs.SMALL.with_(**kw)
    return cfg, inputs.make_activations(cfg), inputs.make_weights(cfg)


def test_x_zero_gives_zero_shared_output():
    cfg, act, w = _small()
    act["x"] = torch.zeros_like(act["x"])
    o = T.tail(act, w, cfg)
    assert np.abs(o["s"]).max() == 0.0
    np.testing.assert_array_equal(o["out"], o["up"])


def test_all_experts_selected_is_softmax_weighted_sum():
    cfg, act, w = _small(E=4, topk=4)
    o = T.tail(act, w, cfg)
    lg = torch.from_numpy(act["logits"].numpy()).double()
    pw = torch.softmax(lg, 1).numpy()
    zd = T.dequant_act(o["zq"], o["zs"])
    ref = np.zeros_like(o["r"])
    for e in range(4):
        w13 = T.dequant_fp8_blocks(w["w13_q"][e], w["w13_s"][e])
        w2 = T.dequant_fp8_blocks(w["w2_q"][e], w["w2_s"][e])
        h = zd @ w13.T
        a = T.silu(h[:, :cfg.I]) * h[:, cfg.I:]
        q, s = T.quant_per128(a.astype(np.float32))
        ref += pw[:, e:e + 1] * (T.dequant_act(q, s) @ w2.T)
    np.testing.assert_allclose(o["r"], ref, rtol=1e-12, atol=1e-12)


def test_one_hot_router_is_single_dense_expert():
    cfg, act, w = _small()
    lg = act["logits"].clone()
    lg[:, 3] = 1e4  # expert 3 always first, with weight 1 to float64 precision
    lg[:, 0] = 1e3
    act["logits"] = lg
    cfg1 = cfg.with_(topk=2)
    o = T.tail(act, w, cfg1)
    assert (o["ids"][:, 0] == 3).all()
    zd = T.dequant_act(o["zq"], o["zs"])
    w13 = torch.from_numpy(T.dequant_fp8_blocks(w["w13_q"][3], w["w13_s"][3]))
    w2 = torch.from_numpy(T.dequant_fp8_blocks(w["w2_q"][3], w["w2_s"][3]))
    h = F.linear(torch.from_numpy(zd), w13)
    a = (F.silu(h[:, :cfg.I]) * h[:, cfg.I:]).numpy()
    q, s = T.quant_per128(a.astype(np.float32))
    ref = F.linear(torch.from_numpy(T.dequant_act(q, s)), w2).numpy()
    np.testing.assert_allclose(o["r"], ref, rtol=1e-12, atol=1e-12)


def test_identity_up_projection_reduces_to_norm():
    cfg, act, w = _small(H=256, L=256)
    w["w_up"] = torch.eye(256, dtype=torch.bfloat16)
    w["gamma"] = torch.ones(256, dtype=torch.bfloat16)
    act["x"] = torch.zeros_like(act["x"])
    o = T.tail(act, w, cfg)
    ref = F.rms_norm(torch.from_numpy(o["r"]), (256,), eps=cfg.eps).numpy()
    np.testing.assert_allclose(o["out"], ref, rtol=1e-12, atol=1e-12)


def test_token_subset_equals_full_rows():
    cfg, act, w = _small(M=9)
    full = T.tail(act, w, cfg)
    sub = T.tail(act, w, cfg, tokens=[7, 2, 4])
    for key in ("out", "r", "s", "n"):  # BLAS blocking differs with the row count
        np.testing.assert_allclose(sub[key], full[key][[7, 2, 4]], rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(sub["zq"], full["zq"][[7, 2, 4]])


# ------------------------------------------------------------------ brute force

@pytest.mark.parametrize("kw", [
    dict(),                                   # M=6, H=L=256, E=4, k=2, I=Is=128
    dict(M=2, E=5, topk=3, seed=12),
    dict(M=3, E=4, topk=4, H=128, L=256, seed=13),
    dict(M=2, E=3, topk=1, H=256, L=128, I=256, seed=14),
])
def test_tail_matches_scalar_brute_force(kw):
    cfg, act, w = _small(**kw)
    o = T.tail(act, w, cfg)
    lg = act["logits"].numpy()
    z = T.to_f64(act["z"])
    x = T.to_f64(act["x"])
    experts = {}
    for e in range(cfg.E):
        experts[e] = (T.dequant_fp8_blocks(w["w13_q"][e], w["w13_s"][e]).tolist(),
                      T.dequant_fp8_blocks(w["w2_q"][e], w["w2_s"][e]).tolist())
    gamma = T.to_f64(w["gamma"]).tolist()
    ws13, ws2, wup = (T.to_f64(w[k]).tolist() for k in ("ws13", "ws2", "w_up"))
    for t in range(cfg.M):
        ref, order, wts = brute.tail_token([float(v) for v in lg[t]], z[t].tolist(),
                                           x[t].tolist(), cfg.topk, experts, gamma, cfg.eps,
                                           ws13, ws2, wup)
        assert o["ids"][t].tolist() == order
        np.testing.assert_allclose(o["w"][t], wts, rtol=1e-13)
        np.testing.assert_allclose(o["out"][t], ref, rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------- the step before the tail

def test_bf16_round_matches_significand_rule_and_ties_to_even():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-8, 8, 2000),
                        [0.0, -0.0, 1.0, -3.5, 1e-30]])
    got = T.bf16_round(v)
    want = np.array([brute.bf16_value(float(a)) for a in v])
    np.testing.assert_array_equal(got, want)
    # exact halfway points between neighbouring bf16 values go to the even significand
    for b in [1.0, 1.0078125, 3.0, -5.0, 0.15625, 255.0]:  # bf16-representable
        ulp = 2.0 ** (np.floor(np.log2(abs(b))) - 7)
        h = b + np.sign(b) * ulp / 2  # halfway to the next bf16 value away from zero
        r = T.bf16_round(np.array([h]))[0]
        assert r in (b, b + np.sign(b) * ulp), (b, r)
        sig = abs(r) / 2.0 ** np.floor(np.log2(abs(r))) * 128  # 8-bit significand
        assert float(sig).is_integer() and int(sig) % 2 == 0, (b, r)


def test_latent_inputs_match_scalar_brute_force():
    rng = np.random.default_rng(8)
    H, L, E, M = 64, 32, 8, 3
    x = torch.from_numpy(rng.standard_normal((M, H)).astype(np.float32)).to(torch.bfloat16)
    w_lat = torch.from_numpy((rng.standard_normal((L, H)) / 8).astype(np.float32)).to(
        torch.bfloat16)
    w_gate = torch.from_numpy((rng.standard_normal((E, H)) / 8).astype(np.float32)).to(
        torch.bfloat16)
    z, lg = T.latent_inputs(x, w_lat, w_gate)
    xs, wl, wg = (t.to(torch.float64).tolist() for t in (x, w_lat, w_gate))
    for t in range(M):
        zb, lb = brute.latent_inputs_token(xs[t], wl, wg)
        np.testing.assert_array_equal(z[t], np.array(zb))
        np.testing.assert_allclose(lg[t], np.array(lb), rtol=1e-13, atol=1e-13)


def test_latent_inputs_zero_and_linear_in_x():
    rng = np.random.default_rng(9)
    H, L, E = 32, 16, 4
    w_lat = rng.standard_normal((L, H))
    w_gate = rng.standard_normal((E, H))
    z0, l0 = T.latent_inputs(np.zeros((2, H)), w_lat, w_gate)
    assert not z0.any() and not l0.any()
    x = rng.standard_normal((3, H))
    _, l1 = T.latent_inputs(x, w_lat, w_gate)
    _, l2 = T.latent_inputs(4.0 * x, w_lat, w_gate)
    np.testing.assert_allclose(l2, 4.0 * l1, rtol=1e-12)
    z1, _ = T.latent_inputs(x, w_lat, w_gate)
    z2, _ = T.latent_inputs(4.0 * x, w_lat, w_gate)  # power-of-two scaling commutes with bf16
    np.testing.assert_array_equal(z2, 4.0 * z1)


# ---------------------------------------------------------------- power-of-two (MX) scales

def _mx_blocks(seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((6, 256)).astype(np.float32)
    v[0] *= 1e-6                       # small magnitudes
    v[1] *= 3e4                        # large magnitudes (quotients reach the e4m3 top)
    v[2, :32] = 0.0                    # an all-zero block
    v[3, 32:64] = np.float32(2.0 ** -20)  # a constant block at an exact power of two
    v[4, 64:96] *= 2.0 ** 40
    return v


def test_quant_mx_matches_scalar_rule():
    v = _mx_blocks(21)
    q, sb = T.quant_mx(v)
    for r in range(v.shape[0]):
        for g in range(v.shape[1] // 32):
            codes, s = brute.quant_group_mx([float(a) for a in v[r, 32 * g:32 * g + 32]])
            assert q[r, 32 * g:32 * g + 32].tolist() == codes, (r, g)
            assert 2.0 ** (int(sb[r, g]) - 127) == s, (r, g)


def test_quant_mx_scale_and_range_properties():
    v = _mx_blocks(22)
    q, sb = T.quant_mx(v)
    d = T.dequant_mx(q, sb)
    for r in range(v.shape[0]):
        for g in range(v.shape[1] // 32):
            blk = v[r, 32 * g:32 * g + 32].astype(np.float64)
            amax = np.abs(blk).max()
            if amax == 0:
                assert sb[r, g] == 127 and not q[r, 32 * g:32 * g + 32].any()
                continue
            e = int(np.floor(np.log2(amax)))
            assert int(sb[r, g]) == e - 8 + 127
            # the block maximum lands in [256, 448] after scaling (saturating above 448)
            top = np.abs(d[r, 32 * g:32 * g + 32]).max() / 2.0 ** (e - 8)
            assert 256.0 <= top <= 448.0
            # per element error: half an e4m3 step, or the saturation at 448
            err = np.abs(d[r, 32 * g:32 * g + 32] - blk)
            assert (err <= np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** (e - 8 - 9)) +
                    np.maximum(np.abs(blk) - 448 * 2.0 ** (e - 8), 0)).all()
    # scaling a row by a power of two shifts the scale bytes and keeps the codes
    q2, sb2 = T.quant_mx(v[5:6] * np.float32(2.0 ** 5))
    np.testing.assert_array_equal(q2, q[5:6])
    np.testing.assert_array_equal(sb2.astype(int), sb[5:6].astype(int) + 5)


def test_dequant_mx_matches_loops():
    rng = np.random.default_rng(23)
    q = rng.integers(0, 256, (3, 64)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0  # no NaN codes
    sb = rng.integers(100, 150, (3, 2)).astype(np.uint8)
    d = T.dequant_mx(q, sb)
    for r in range(3):
        for c in range(64):
            assert d[r, c] == brute.e4m3_value(int(q[r, c])) * 2.0 ** (int(sb[r, c // 32]) - 127)


def test_generator_mx_roundtrip_of_representable_weights():
    # weights that are e4m3 values times a power of two per block are stored exactly
    rng = np.random.default_rng(24)
    codes = rng.integers(0, 0x7F, (128, 64)).astype(np.uint8)
    codes[:, ::32] = 0x7E  # each block holds 448 (its maximum)
    sign = np.where(rng.random((128, 64)) < 0.5, -1.0, 1.0)
    scale = 2.0 ** rng.integers(-20, 5, (128, 2))
    w = np.array([[brute.e4m3_value(int(c)) for c in row] for row in codes]) * sign
    w = w * np.repeat(scale, 32, axis=1)
    q, sb = inputs.mx_quantize(torch.from_numpy(w.astype(np.float32)))
    np.testing.assert_array_equal(T.dequant_mx(q.numpy(), sb.numpy()), w)


@pytest.mark.parametrize("kw", [dict(), dict(M=2, E=5, topk=3, seed=12)])
def test_tail_mx_matches_scalar_brute_force(kw):
    cfg, act, w = _small(routed_fmt="mxfp8", **kw)
    o = T.tail(act, w, cfg)
    lg = act["logits"].numpy()
    z = T.to_f64(act["z"])
    x = T.to_f64(act["x"])
    experts = {e: (T.dequant_mx(w["w13_q"][e].numpy(), w["w13_sx"][e].numpy()).tolist(),
                   T.dequant_mx(w["w2_q"][e].numpy(), w["w2_sx"][e].numpy()).tolist())
               for e in range(cfg.E)}
    gamma = T.to_f64(w["gamma"]).tolist()
    ws13, ws2, wup = (T.to_f64(w[k]).tolist() for k in ("ws13", "ws2", "w_up"))
    for t in range(cfg.M):
        ref, order, wts = brute.tail_token([float(v) for v in lg[t]], z[t].tolist(),
                                           x[t].tolist(), cfg.topk, experts, gamma, cfg.eps,
                                           ws13, ws2, wup, mx=True)
        assert o["ids"][t].tolist() == order
        np.testing.assert_allclose(o["out"][t], ref, rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------- NVFP4 activations (FP4 x FP4)

def test_e2m1_encode_matches_nearest_value_search():
    from oracle.codecs import e2m1_encode
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])]
    rng = np.random.default_rng(31)
    vals = grid + mids + [6.5, 1e9, 1e-30] + list(rng.uniform(-7, 7, 400))
    vals += [-v for v in vals]
    got = e2m1_encode(np.array(vals)).tolist()
    assert got == [brute.e2m1_round(v) for v in vals]
    # ties go to the even code: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    assert e2m1_encode(np.array(mids)).tolist() == [0, 2, 2, 4, 4, 6, 6]
    # every code decodes and re-encodes to itself (negative zero excepted: it has code 0)
    from oracle.codecs import e2m1_decode
    codes = np.array([c for c in range(16) if c != 8])
    assert e2m1_encode(e2m1_decode(codes)).tolist() == codes.tolist()


def _nv_blocks(seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((6, 128)).astype(np.float32)
    v[0] *= 1e-4                        # scales in the e4m3 subnormal range
    v[1] *= 2e3                         # amax / 6 above 448: the scale saturates
    v[2, :16] = 0.0                     # an all-zero block
    v[2, 16:32] = np.float32(1e-5)      # amax / 6 rounds to a zero scale
    v[3, 32:48] = np.float32(3.0)       # a constant block
    v[4, 48:64] *= 2.0 ** 6
    return v


def test_quant_nvfp4_matches_scalar_rule():
    v = _nv_blocks(32)
    q, sb = T.quant_nvfp4(v)
    for r in range(v.shape[0]):
        for g in range(v.shape[1] // 16):
            codes, s = brute.quant_group_nvfp4([float(a) for a in v[r, 16 * g:16 * g + 16]])
            assert q[r, 16 * g:16 * g + 16].tolist() == codes, (r, g)
            assert float(e4m3_decode(sb[r, g])) == s, (r, g)


def test_quant_nvfp4_scale_and_range_properties():
    v = _nv_blocks(33)
    q, sb = T.quant_nvfp4(v)
    d = T.dequant_nvfp4_act(q, sb)
    s = e4m3_decode(sb)
    assert sb[2, 0] == 0 and sb[2, 1] == 0 and not q[2, :32].any()
    assert (sb[1] == 0x7E).all()        # saturated scales: 448
    for r in (3, 4, 5):                 # normal-range blocks
        for g in range(8):
            blk = v[r, 16 * g:16 * g + 16].astype(np.float64)
            amax = np.abs(blk).max()
            # the scale is amax / 6 to within half an e4m3 step, so the block maximum
            # lands on the top code 6 (code 7), saturating when the scale rounded down
            assert abs(s[r, g] - amax / 6) <= s[r, g] * 2.0 ** -4
            assert (q[r, 16 * g:16 * g + 16] & 7).max() == 7
            # per element error: half the local e2m1 spacing (at most 1 in scaled units)
            # plus the saturation at 6
            err = np.abs(d[r, 16 * g:16 * g + 16] - blk)
            assert (err <= s[r, g] * 1.0 + np.maximum(np.abs(blk) - 6 * s[r, g], 0) + 1e-12).all()
    # scaling a row by a power of two moves each normal scale's exponent, codes unchanged
    q2, sb2 = T.quant_nvfp4(v[5:6] * np.float32(2.0 ** 3))
    np.testing.assert_array_equal(q2, q[5:6])
    np.testing.assert_array_equal(sb2.astype(int), sb[5:6].astype(int) + (3 << 3))


def test_dequant_nvfp4_act_matches_loops():
    rng = np.random.default_rng(34)
    q = rng.integers(0, 16, (3, 32)).astype(np.uint8)
    sb = rng.integers(0, 0x7F, (3, 2)).astype(np.uint8)
    d = T.dequant_nvfp4_act(q, sb)
    for r in range(3):
        for c in range(32):
            assert d[r, c] == brute.e2m1_value(int(q[r, c])) * brute.e4m3_value(int(sb[r, c // 16]))


@pytest.mark.parametrize("kw", [dict(), dict(M=2, E=5, topk=3, seed=13)])
def test_tail_w4a4_matches_scalar_brute_force(kw):
    cfg, act, w = _small(routed_fmt="nvfp4_w4a4", **kw)
    o = T.tail(act, w, cfg)
    lg = act["logits"].numpy()
    z = T.to_f64(act["z"])
    x = T.to_f64(act["x"])
    experts = {e: (T.dequant_nvfp4(w["w13_q"][e], w["w13_sb"][e], float(w["w13_g"][e])).tolist(),
                   T.dequant_nvfp4(w["w2_q"][e], w["w2_sb"][e], float(w["w2_g"][e])).tolist())
               for e in range(cfg.E)}
    gamma = T.to_f64(w["gamma"]).tolist()
    ws13, ws2, wup = (T.to_f64(w[k]).tolist() for k in ("ws13", "ws2", "w_up"))
    for t in range(cfg.M):
        ref, order, wts = brute.tail_token([float(v) for v in lg[t]], z[t].tolist(),
                                           x[t].tolist(), cfg.topk, experts, gamma, cfg.eps,
                                           ws13, ws2, wup, a4=True)
        assert o["ids"][t].tolist() == order
        np.testing.assert_allclose(o["out"][t], ref, rtol=1e-9, atol=1e-9)
    # the latent codes are the quantiser's own (one e2m1 code per element)
    q, sb = T.quant_nvfp4(z.astype(np.float32))
    np.testing.assert_array_equal(o["zq"], q)
    np.testing.assert_array_equal(o["zs"], sb)
