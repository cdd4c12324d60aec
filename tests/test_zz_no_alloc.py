"""klt_route_noalloc, the allocation-free routing entry point, against klt_forward and
the float64 oracle.

Some callers cannot allocate device memory where they route (they run inside another
framework's memory pool, or pin every allocation at start-up); klt_route_noalloc serves
them with a fixed internal scratch array.  Its routing and permutation outputs must equal
the ones klt_forward reports for the same logits, on consecutive calls that reuse the
shared scratch.  This file is collected last so that a failure here never hides the other
tests' results; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from latent_moe_layer_route_gb300 import binding as B
from latent_moe_layer_route_gb300 import build, configs, inputs
from oracle import model as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    B.load_library()


def _routing_buffers(M, E, k):
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(ids=torch.full((M, k), -1, **i32),
                weights=torch.full((M, k), float("nan"), dtype=torch.float32, device="cuda"),
                cnt=torch.full((E,), -1, **i32), off=torch.full((E + 1,), -1, **i32),
                gidx=torch.full((M * k,), -1, **i32), slot=torch.full((M * k,), -1, **i32),
                pos=torch.full((M, k), -1, **i32))


def _via_forward(cfg, act, w_gpu):
    M = act["x"].shape[0]
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=M)
    try:
        buf = _routing_buffers(M, cfg.E, cfg.topk)
        ro = B.KltRouting(*(buf[n].data_ptr() for n in
                            ("ids", "weights", "cnt", "off", "gidx", "slot", "pos")))
        tail.forward(act["x"], act["z"], act["logits"], routing=ro)
        torch.cuda.synchronize()
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()
    return buf


def _via_noalloc(logits, k):
    M, E = logits.shape
    buf = _routing_buffers(M, E, k)
    rc = B.klt_route_noalloc(logits, k, buf["ids"], buf["weights"], buf["cnt"], buf["off"],
                             buf["gidx"], buf["slot"], buf["pos"],
                             torch.cuda.current_stream().cuda_stream)
    assert rc == B.KLT_OK, B.strerror(rc)
    torch.cuda.synchronize()
    return buf


def _same(a, b):
    for name in ("ids", "cnt", "off", "gidx", "slot", "pos"):
        assert torch.equal(a[name], b[name]), name
    torch.testing.assert_close(a["weights"], b["weights"], rtol=1e-6, atol=1e-7)


def _matches_oracle(buf, logits, k, E):
    ids, w = T.route(logits.cpu().numpy(), k)
    np.testing.assert_array_equal(buf["ids"].cpu().numpy(), ids)
    np.testing.assert_allclose(buf["weights"].cpu().numpy().astype(np.float64), w, rtol=1e-6,
                               atol=1e-7)
    for name, ref in zip(("cnt", "off", "gidx", "slot", "pos"), T.permutation(ids, E)):
        np.testing.assert_array_equal(buf[name].cpu().numpy(), ref, err_msg=name)


# one and two permutation blocks (k = 2), and exactly the scratch capacity: 8192 tokens x
# top-8 = KLT_NOALLOC_MAX_PAIRS pairs, 64 permutation blocks in the histogram region
@pytest.mark.parametrize("M,E,k", [(37, 8, 2), (700, 8, 2), (8192, 64, 8)])
def test_noalloc_routing_matches_forward_on_two_calls_in_a_row(M, E, k):
    cfg = configs.SMALL.with_(E=E, topk=k, seed=31)
    assert M * k <= B.KLT_NOALLOC_MAX_PAIRS
    w_gpu = {n: v.cuda() for n, v in inputs.make_weights(cfg).items()}
    act = {n: v.cuda() for n, v in inputs.make_activations(cfg, M).items()}
    ref = _via_forward(cfg, act, w_gpu)
    first = _via_noalloc(act["logits"], cfg.topk)
    second = _via_noalloc(act["logits"], cfg.topk)
    _same(first, ref)
    _same(second, ref)
    _matches_oracle(second, act["logits"], k, E)


def test_noalloc_accepts_exactly_its_capacity_and_rejects_one_more_pair():
    E = 8
    rng = np.random.default_rng(3)
    logits = torch.from_numpy(
        rng.standard_normal((B.KLT_NOALLOC_MAX_PAIRS + 1, E), dtype=np.float32)).cuda()
    full = logits[:B.KLT_NOALLOC_MAX_PAIRS]
    got = _via_noalloc(full, 1)
    _matches_oracle(got, full, 1, E)
    buf = _routing_buffers(B.KLT_NOALLOC_MAX_PAIRS + 1, E, 1)
    rc = B.klt_route_noalloc(logits, 1, buf["ids"], buf["weights"], buf["cnt"], buf["off"],
                             buf["gidx"], buf["slot"], buf["pos"])
    assert rc == B.KLT_ERR_TOO_LARGE


def test_noalloc_rejects_requests_beyond_its_scratch():
    logits = torch.zeros((B.KLT_NOALLOC_MAX_PAIRS // 2 + 1, 8), dtype=torch.float32,
                         device="cuda")
    buf = _routing_buffers(1, 8, 2)
    rc = B.klt_route_noalloc(logits, 2, buf["ids"], buf["weights"], buf["cnt"], buf["off"],
                             buf["gidx"], buf["slot"], buf["pos"])
    assert rc == B.KLT_ERR_TOO_LARGE
    assert "scratch" in B.strerror(rc)
