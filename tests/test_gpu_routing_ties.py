"""The router's tie rule on the GPU, bit for bit against the float64 oracle.

Routing picks each token's k largest logits; equal logits go to the lower expert index,
and -0.0 equals +0.0.  Random normal logits almost never tie, so these cases build ties
on purpose: all-zero rows, logits on a coarse grid (many ties straddle the top-k
boundary), rows mixing -0.0 and +0.0, and the widest router (256 experts, top-32).  The
routing arrays (ids, cnt, off, gidx, slot, pos) must equal the oracle's exactly, the
weights within 1e-6, through klt_forward on both GEMM engines' token ranges and through
klt_route_noalloc."""
import numpy as np
import pytest
import torch

from latent_moe_layer_route_gb300 import binding as B
from latent_moe_layer_route_gb300 import build, configs, inputs
from oracle import model as T
import parity_util as PU

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    B.load_library()


def _grid_logits(M, E, seed, step=0.25):
    rng = np.random.default_rng(seed)
    return (np.round(rng.standard_normal((M, E)) / step) * step).astype(np.float32)


def _signed_zero_logits(M, E, seed):
    # every row: a few positive logits, then -0.0 / +0.0 mixed, the rest negative, so the
    # top-k boundary falls inside the run of zeros of both signs
    rng = np.random.default_rng(seed)
    lg = -1.0 - rng.random((M, E)).astype(np.float32)
    for t in range(M):
        cols = rng.permutation(E)
        lg[t, cols[:3]] = 1.0 + rng.random(3).astype(np.float32)
        zeros = cols[3:3 + E // 2]
        lg[t, zeros] = np.where(rng.random(len(zeros)) < 0.5, -0.0, 0.0).astype(np.float32)
    assert np.signbit(lg[lg == 0]).any() and (~np.signbit(lg[lg == 0])).any()
    return lg


def _logits(kind, M, E, seed):
    if kind == "zero":
        return np.zeros((M, E), dtype=np.float32)
    if kind == "grid":
        return _grid_logits(M, E, seed)
    return _signed_zero_logits(M, E, seed)


def _check_routing_exact(ids, w, cnt, off, gidx, slot, pos, logits, k, E):
    r_ids, r_w = T.route(logits, k)
    np.testing.assert_array_equal(ids, r_ids)
    np.testing.assert_allclose(w.astype(np.float64), r_w, rtol=1e-6, atol=1e-7)
    assert np.abs(w.astype(np.float64).sum(1) - 1.0).max() <= 1e-6
    r_cnt, r_off, r_gidx, r_slot, r_pos = T.permutation(r_ids, E)
    for got, ref in ((cnt, r_cnt), (off, r_off), (gidx, r_gidx), (slot, r_slot),
                     (pos, r_pos)):
        np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("kind", ["zero", "grid", "signed_zero"])
@pytest.mark.parametrize("M,bn", [(16, 16), (300, 256)])  # feature-major / token-major range
def test_forward_routing_ties(kind, M, bn):
    cfg = configs.SMALL.with_(E=64, topk=8, seed=51)
    w_cpu = inputs.make_weights(cfg)
    w_gpu = PU.to_cuda(w_cpu)
    act = inputs.make_activations(cfg, M)
    lg = _logits(kind, M, cfg.E, seed=M)
    act["logits"] = torch.from_numpy(lg)
    if kind == "grid":  # ties must actually cross the top-k boundary
        srt = -np.sort(-lg, axis=1)
        assert (srt[:, cfg.topk - 1] == srt[:, cfg.topk]).sum() > M // 4
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=M)
    try:
        assert tail.gemm_tile(M) == bn
        run = PU.Run(tail, PU.to_cuda(act), cfg)
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()
    _check_routing_exact(*(run.host(n).numpy() for n in
                           ("ids", "w", "cnt", "off", "gidx", "slot", "pos")), lg, cfg.topk,
                         cfg.E)
    if kind == "zero":  # every token picks experts 0..k-1 with weight 1/k
        ids = run.host("ids").numpy()
        assert (ids == np.arange(cfg.topk)[None, :]).all()
        assert (run.host("w").numpy() == np.float32(1.0 / cfg.topk)).all()
    # the whole tail still meets the output bar on the tied routing
    o = T.tail(act, w_cpu, cfg, tokens=np.arange(min(M, 24)))
    PU.check_stages(run, o, cfg)


@pytest.mark.parametrize("bn", [16, 256])
def test_forward_ties_widest_router_256_experts_top32(bn):
    cfg = configs.SMALL.with_(E=256, topk=32, seed=52)
    M = 20
    w_cpu = inputs.make_weights(cfg)
    act = inputs.make_activations(cfg, M)
    lg = _grid_logits(M, cfg.E, seed=5, step=0.5)
    act["logits"] = torch.from_numpy(lg)
    tail = B.LatentMoETail(cfg, PU.to_cuda(w_cpu), max_tokens=M)
    try:
        run = PU.Run(tail, PU.to_cuda(act), cfg, force_bn=bn)
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()
    _check_routing_exact(*(run.host(n).numpy() for n in
                           ("ids", "w", "cnt", "off", "gidx", "slot", "pos")), lg, cfg.topk,
                         cfg.E)


@pytest.mark.parametrize("kind", ["zero", "grid", "signed_zero"])
@pytest.mark.parametrize("M,E,k", [(300, 64, 8), (20, 256, 32), (3000, 64, 8)])
def test_noalloc_routing_ties(kind, M, E, k):
    lg = _logits(kind, M, E, seed=M + E)
    d = torch.from_numpy(lg).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    buf = dict(ids=torch.full((M, k), -1, **i32),
               w=torch.full((M, k), float("nan"), dtype=torch.float32, device="cuda"),
               cnt=torch.full((E,), -1, **i32), off=torch.full((E + 1,), -1, **i32),
               gidx=torch.full((M * k,), -1, **i32), slot=torch.full((M * k,), -1, **i32),
               pos=torch.full((M, k), -1, **i32))
    rc = B.klt_route_noalloc(d, k, buf["ids"], buf["w"], buf["cnt"], buf["off"], buf["gidx"],
                             buf["slot"], buf["pos"], torch.cuda.current_stream().cuda_stream)
    assert rc == B.KLT_OK, B.strerror(rc)
    torch.cuda.synchronize()
    _check_routing_exact(*(buf[n].cpu().numpy() for n in
                           ("ids", "w", "cnt", "off", "gidx", "slot", "pos")), lg, k, E)
