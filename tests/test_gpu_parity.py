"""CUDA path vs the float64 oracle, through the C ABI, on seeded synthetic inputs.

Index and permutation outputs and the latent quantisation must match bit for bit; float
stages must meet the tail's bar (relative Frobenius error <= 5e-3 and per element
|err| <= 0.03*rms(ref) + 0.01*|ref|)."""
import numpy as np
import pytest
import torch

from latent_moe_layer_route_gb300 import binding as B
from latent_moe_layer_route_gb300 import build, configs, inputs
from oracle import model as T
import parity_util as PU

pytestmark = pytest.mark.gpu

_CACHE = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    B.load_library()
    yield
    _CACHE.clear()


def weights_for(cfg):
    key = (cfg.E, cfg.topk, cfg.I, cfg.H, cfg.L, cfg.Is, cfg.routed_fmt, cfg.seed)
    if key not in _CACHE:
        _CACHE.clear()
        w = inputs.make_weights(cfg)
        _CACHE[key] = (w, PU.to_cuda(w))
    return _CACHE[key]


def run_case(cfg, M=None, act=None, tokens=None, max_tokens=None, tail=None, force_bn=0,
             flags=0, expect_tile=None):
    w_cpu, w_gpu = weights_for(cfg)
    if act is None:
        act = inputs.make_activations(cfg, M)
    M = act["x"].shape[0]
    own = tail is None
    if own:
        tail = B.LatentMoETail(cfg, w_gpu, max_tokens=max_tokens or M, flags=flags)
    # the engine under test is the one the library runs
    tile = tail.gemm_tile(M, force_bn)
    assert tile == (expect_tile if expect_tile is not None else (force_bn or tile))
    run = PU.Run(tail, PU.to_cuda(act), cfg, force_bn=force_bn)
    assert tail.status() == B.KLT_OK
    o = T.tail(act, w_cpu, cfg, tokens=tokens)
    PU.check_routing(run, o, cfg)
    rf = PU.check_stages(run, o, cfg, combine_buffer=not flags & B.KLT_FLAG_DETERMINISTIC)
    if own:
        tail.close()
    return run, o, rf


# ------------------------------------------------------------------ small shapes

@pytest.mark.parametrize("M", [1, 6, 17, 40])
def test_small_shapes(M):
    run_case(configs.SMALL, M=M)


@pytest.mark.parametrize("M", [3, 33])
def test_small_nvfp4(M):
    run_case(configs.SMALL.with_(routed_fmt="nvfp4", E=6, topk=2, seed=28), M=M)


def test_small_nvfp4_wider():
    run_case(configs.SMALL.with_(routed_fmt="nvfp4", H=384, L=512, I=256, Is=256, E=5,
                                 topk=3, seed=29), M=45)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("M", [3, 9])
def test_routed_l1_k_split(fmt, M):
    # few touched experts: the routed L1 units are split in K (two splits of whole promotion
    # groups), the last split of each tile sums the partials and runs the epilogue
    cfg = configs.SMALL.with_(L=1024, E=4, topk=2, routed_fmt=fmt, seed=41)
    run_case(cfg, M=M, force_bn=16)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("M,topk,L,launches", [
    (16, 16, 256, 2),  # 256 pairs: the most the one-launch routing takes
    (5, 3, 640, 2),    # five 128-column groups: a partial group batch per warp
    (17, 16, 640, 4),  # 272 pairs: routing, scatter and gather launches
])
def test_one_launch_routing_at_its_pair_limit(fmt, M, topk, L, launches):
    # a feature-major batch of at most 256 (token, choice) pairs is routed, sorted and
    # quantised into expert order by one launch; one pair more takes the three-launch chain
    cfg = configs.SMALL.with_(routed_fmt=fmt, E=64, topk=topk, L=L, seed=39)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=M)
    try:
        assert tail.gemm_tile(M, 0) != 256
        assert tail.launch_count(M) == launches
        run_case(cfg, M=M, tail=tail)
    finally:
        tail.close()


@pytest.mark.parametrize("bn", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_every_token_tile_width(bn, fmt):
    # ragged M spanning several token tiles of each width (256: the token-major engine)
    run_case(configs.SMALL.with_(routed_fmt=fmt, E=6, topk=3, seed=30), M=150, force_bn=bn)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_token_major_engine_on_several_feature_tiles(fmt):
    # two routed L1 tiles, two L2 and three output tiles of 256 features, two shared L1
    # tiles, ragged 128-token tiles of 8 experts
    cfg = configs.SMALL.with_(routed_fmt=fmt, H=768, L=512, I=256, Is=256, E=8, topk=2,
                              seed=33)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=300)
    try:
        assert tail.gemm_tile(300, 256) == 256
        run_case(cfg, M=300, tail=tail, force_bn=256)
    finally:
        tail.close()


@pytest.mark.parametrize("M", [17, 200])
def test_token_major_output_split_in_k(M):
    # one or two token tiles (the second ragged): the output GEMM runs as k-splits that add
    # into fp32 tiles, the last split of each tile rounding it; a second forward on the
    # same handle finds the tiles and their counters reset
    cfg = configs.SMALL.with_(H=1024, L=1024, I=256, Is=512, E=8, topk=2, seed=40)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=M)
    try:
        assert tail.gemm_tile(M, 256) == 256
        for _ in range(2):
            run_case(cfg, M=M, tail=tail, force_bn=256)
    finally:
        tail.close()


def test_token_major_engine_with_long_k():
    # a small batch with long K: the output GEMM's k loop crosses from the up-projection
    # into the shared down projection far from the first k-block
    cfg = configs.SMALL.with_(H=2048, L=1024, I=256, Is=256, E=8, topk=2, seed=36)
    run_case(cfg, M=40, force_bn=256)


@pytest.mark.parametrize("bn", [16, 256])
def test_largest_router_256_experts_top32(bn):
    # the router's widest expert set and deepest top-k, on both GEMM engines
    cfg = configs.SMALL.with_(E=256, topk=32, seed=37)
    run_case(cfg, M=20, force_bn=bn)


@pytest.mark.slow
@pytest.mark.parametrize("bn", [16, 256])
def test_longest_latent_and_intermediate_4096(bn):
    # L = I = 4096: 32 k-blocks per routed unit, the most the engines stage per unit
    cfg = configs.SMALL.with_(L=4096, I=4096, E=2, topk=2, seed=38)
    run_case(cfg, M=24, force_bn=bn)


def test_token_major_engine_dual_token_tiles():
    # from 16 token tiles on, the shared L1 and output units take two token tiles each
    # (3 stages of 64 KB): 17 tiles, the last one ragged and unpaired
    cfg = configs.SMALL.with_(E=8, topk=2, seed=39)
    rng = np.random.default_rng(2)
    tok = np.sort(np.concatenate([rng.choice(2048, 40, replace=False), np.arange(2048, 2100)]))
    run_case(cfg, M=2100, tokens=tok, force_bn=256)


def test_token_major_engine_is_chosen_above_the_decode_tile():
    cfg = configs.SMALL.with_(seed=34)
    _, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=2048)
    phased = B.LatentMoETail(cfg, w_gpu, max_tokens=2048, flags=B.KLT_FLAG_PHASED)
    try:
        assert tail.gemm_tile(2048) == 256 and tail.gemm_tile(17) == 256
        assert tail.gemm_tile(16) == 16 and tail.gemm_tile(1) == 16
        assert tail.gemm_tile(16, 128) == 128
        assert phased.gemm_tile(2048) == 64
        assert phased.gemm_tile(2048, 256) == -B.KLT_ERR_UNSUPPORTED
    finally:
        tail.close()
        phased.close()
    narrow = configs.SMALL.with_(H=384, seed=35)  # H not a multiple of 256
    _, w_gpu = weights_for(narrow)
    tail = B.LatentMoETail(narrow, w_gpu, max_tokens=2048)
    try:
        assert tail.gemm_tile(2048) == 64
        assert tail.gemm_tile(8, 256) == -B.KLT_ERR_UNSUPPORTED
    finally:
        tail.close()


@pytest.mark.parametrize("bn", [16, 64])
@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_phased_launches_match_the_oracle_too(bn, fmt):
    # the three-launch schedule (one GEMM launch per stage) computes the same tail
    run_case(configs.SMALL.with_(routed_fmt=fmt, E=6, topk=3, seed=32), M=70, force_bn=bn,
             flags=B.KLT_FLAG_PHASED)


def test_small_all_experts_selected():
    run_case(configs.SMALL.with_(E=4, topk=4, seed=21), M=9)


def test_small_wider_k_tail_shapes():
    # several 128-tiles in every dimension and a ragged token count
    run_case(configs.SMALL.with_(H=512, L=384, I=256, Is=384, E=8, topk=3, seed=22), M=29)


def test_one_hot_routing_sends_every_token_to_one_expert():
    cfg = configs.SMALL.with_(E=8, topk=2, seed=23)
    act = inputs.make_activations(cfg, 33)
    act["logits"][:, 5] += 50.0
    run, o, _ = run_case(cfg, act=act)
    assert o["cnt"][5] == 33


def test_zero_latent_leaves_shared_expert_only():
    cfg = configs.SMALL.with_(seed=24)
    act = inputs.make_activations(cfg, 8)
    act["z"] = torch.zeros_like(act["z"])
    run, o, _ = run_case(cfg, act=act)
    assert float(run.r.abs().max()) == 0.0


def test_zero_hidden_leaves_routed_branch_only():
    cfg = configs.SMALL.with_(seed=25)
    act = inputs.make_activations(cfg, 8)
    act["x"] = torch.zeros_like(act["x"])
    run, o, _ = run_case(cfg, act=act)
    assert float(run.a_s.float().abs().max()) == 0.0


def test_repeated_calls_and_smaller_m_reuse_the_workspace():
    cfg = configs.SMALL.with_(seed=26)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=64)
    try:
        for M in (64, 5, 64, 33):
            act = inputs.make_activations(cfg, M)
            run = PU.Run(tail, PU.to_cuda(act), cfg)
            o = T.tail(act, w_cpu, cfg)
            PU.check_routing(run, o, cfg)
            PU.check_stages(run, o, cfg)
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()


@pytest.mark.parametrize("M,bn", [(12, 0), (40, 256)])
def test_two_consecutive_forwards_replayed_from_a_cuda_graph(M, bn):
    # two layers' tails captured in one CUDA graph (the launches of each forward, and of the
    # second after the first, chained by programmatic dependent launch edges), replayed
    # twice: every output matches the oracle, and the replays match each other
    cfg = configs.SMALL.with_(E=8, topk=3, seed=44)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=M)
    try:
        acts = [inputs.make_activations(cfg.with_(seed=44 + i), M) for i in range(2)]
        dev = [PU.to_cuda(a) for a in acts]
        outs = [torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        dbg = B.KltDebug()
        dbg.force_bn = bn

        def layers():
            for a, o in zip(dev, outs):
                tail.forward(a["x"], a["z"], a["logits"], out=o, debug=dbg)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            layers()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layers()
        got = []
        for _ in range(2):
            for o in outs:
                o.fill_(0)
            g.replay()
            torch.cuda.synchronize()
            assert tail.status() == B.KLT_OK
            got.append([o.float().cpu().numpy().astype(np.float64) for o in outs])
        for a, y in zip(acts, got[0]):
            PU.assert_output_close(y, T.tail(a, w_cpu, cfg)["out"])
        for y0, y1 in zip(got[0], got[1]):
            assert PU.rel_fro(y1, y0) <= 1e-3  # the fp32 combine adds in arrival order
        del g
    finally:
        tail.close()


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("M,bn", [(12, 0), (40, 256), (300, 256)])
def test_deterministic_combine_matches_the_oracle_and_repeats_bitwise(fmt, M, bn):
    # each (token, choice) slot's weighted output stored, summed in choice order by the norm
    cfg = configs.SMALL.with_(E=8, topk=3, routed_fmt=fmt, seed=45)
    run_case(cfg, M=M, force_bn=bn, flags=B.KLT_FLAG_DETERMINISTIC)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=M, flags=B.KLT_FLAG_DETERMINISTIC)
    try:
        a = PU.to_cuda(inputs.make_activations(cfg, M))
        dbg = B.KltDebug()
        dbg.force_bn = bn
        outs = []
        for _ in range(3):
            outs.append(tail.forward(a["x"], a["z"], a["logits"], debug=dbg).clone())
        torch.cuda.synchronize()
        assert tail.status() == B.KLT_OK
        for o in outs[1:]:
            assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    finally:
        tail.close()


def test_m_zero_is_a_noop_and_bad_m_is_rejected():
    cfg = configs.SMALL
    _, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=8)
    try:
        x = torch.zeros((8, cfg.H), dtype=torch.bfloat16, device="cuda")
        z = torch.zeros((8, cfg.L), dtype=torch.bfloat16, device="cuda")
        lg = torch.zeros((8, cfg.E), dtype=torch.float32, device="cuda")
        out = torch.full((8, cfg.H), 3.0, dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        assert B.klt_forward(tail.handle, x, z, lg, 0, out, stream=s) == B.KLT_OK
        torch.cuda.synchronize()
        assert bool((out == 3.0).all())
        assert B.klt_forward(tail.handle, x, z, lg, 9, out, stream=s) == B.KLT_ERR_INVALID_ARG
        assert B.klt_forward(tail.handle, x, z, lg, -1, out, stream=s) == \
            B.KLT_ERR_INVALID_ARG
        lib = B.load_library()
        assert lib.klt_forward(tail.handle, x.data_ptr() + 2, z.data_ptr(), lg.data_ptr(), 4,
                               out.data_ptr(), None, None, s) == B.KLT_ERR_ALIGN
        assert lib.klt_forward(tail.handle, None, z.data_ptr(), lg.data_ptr(), 4,
                               out.data_ptr(), None, None, s) == B.KLT_ERR_INVALID_ARG
        # one routing launch (a small batch) and the fused GEMM launch
        assert tail.launch_count(4) == 2 and tail.launch_count(0) == 0
    finally:
        tail.close()


@pytest.mark.parametrize("bn", [0, 256])
def test_bounded_wait_expires_into_status_without_faulting(bn):
    cfg = configs.SMALL.with_(seed=27)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=16)
    try:
        act = PU.to_cuda(inputs.make_activations(cfg, 16))
        PU.Run(tail, act, cfg, stall_after=1, timeout_ms=20, force_bn=bn)
        assert tail.status() == B.KLT_ERR_DEVICE_TIMEOUT
        # the context is still usable: a fresh handle runs correctly
        run_case(cfg, M=16, force_bn=bn)
    finally:
        tail.close()


# ------------------------------------------------------------------ the named workloads

def test_tiny_m4():
    _, _, rf = run_case(configs.TINY_M4)
    print("tiny rel_fro", rf)


def test_decode_m16():
    _, _, rf = run_case(configs.DECODE_M16)
    print("decode m16 rel_fro", rf)


def test_decode_m16_phased():
    run_case(configs.DECODE_M16, flags=B.KLT_FLAG_PHASED)


def test_decode_m128():
    _, _, rf = run_case(configs.DECODE_M128)
    print("decode m128 rel_fro", rf)


@pytest.mark.slow
@pytest.mark.parametrize("bn", [0, 64])  # 0: the token-major engine chosen for M=4096
def test_prefill_m4096_sampled_tokens(bn):
    cfg = configs.PREFILL_M4096
    rng = np.random.default_rng(0)
    tok = np.sort(rng.choice(cfg.M, 48, replace=False))
    tok[0], tok[-1] = 0, cfg.M - 1
    run_case(cfg, tokens=tok, force_bn=bn, expect_tile=bn or 256)


@pytest.mark.slow
def test_prefill_m8192_nvfp4_sampled_tokens():
    cfg = configs.PREFILL_M8192_NVFP4
    rng = np.random.default_rng(1)
    tok = np.sort(rng.choice(cfg.M, 32, replace=False))
    tok[0], tok[-1] = 0, cfg.M - 1
    run_case(cfg, tokens=tok, expect_tile=256)


# ------------------------------------------------------------------ combine buffer reuse

@pytest.mark.parametrize("M1,M2,flags,fmt", [(12, 16, 0, "fp8"), (40, 70, 0, "fp8"),
                                             (12, 16, B.KLT_FLAG_PHASED, "fp8"),
                                             (40, 70, 0, "mxfp8")])
def test_combine_buffer_reuse_across_forwards(M1, M2, flags, fmt):
    """The fp32 combine buffer is zeroed by the norm rows for the next forward (not by the
    routing kernel); a forward that copies it out leaves it, and the next one clears it.
    Forwards of growing and shrinking M on one handle, with and without that copy, must
    each match the oracle."""
    cfg = configs.SMALL.with_(routed_fmt=fmt, E=8, topk=3, seed=91)
    w_cpu, w_gpu = weights_for(cfg)
    tail = B.LatentMoETail(cfg, w_gpu, max_tokens=max(M1, M2), flags=flags)
    try:
        plan = [(M1, False), (M2, False), (M1, True), (M2, False), (M1, False)]
        for i, (M, debug) in enumerate(plan):
            act = inputs.make_activations(cfg.with_(seed=100 + i), M)
            o = T.tail(act, w_cpu, cfg)
            if debug:  # copies r out: the next forward clears it first
                run = PU.Run(tail, PU.to_cuda(act), cfg)
                assert tail.status() == B.KLT_OK
                PU.check_stages(run, o, cfg)
            else:
                a = PU.to_cuda(act)
                out = tail.forward(a["x"], a["z"], a["logits"])
                torch.cuda.synchronize()
                assert tail.status() == B.KLT_OK
                PU.assert_output_close(out.float().cpu().numpy().astype(np.float64), o["out"])
    finally:
        tail.close()
