"""The FP4 x FP4 routed format (NVFP4 weights kept packed, NVFP4 activations: e2m1 codes
with an e4m3 scale per 16, applied by the tensor core's block-scaled FP4 MMA) against the
float64 oracle, through the C ABI.

Routing, the permutation, the latent codes and their scale bytes must match bit for bit;
the routed activation codes where the GPU's fp32 accumulation does not move a value across
a rounding boundary; the combine, the normalised latent, the shared activation and the
output within the tail's bar."""
import numpy as np
import pytest
import torch

from latent_moe_layer_route_gb300 import binding as B
from latent_moe_layer_route_gb300 import build, configs, inputs
from oracle import model as T
import parity_util as PU

pytestmark = pytest.mark.gpu

FMT = "nvfp4_w4a4"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    B.load_library()


def _case(cfg, M, tokens=None, flags=0):
    w = inputs.make_weights(cfg)
    act = inputs.make_activations(cfg, M)
    tail = B.LatentMoETail(cfg, PU.to_cuda(w), max_tokens=M, flags=flags)
    try:
        assert tail.gemm_tile(M) == 256  # block-scaled units live in the token-major engine
        assert tail.gemm_tile(M, 16) == -B.KLT_ERR_UNSUPPORTED
        assert tail.launch_count(M) == 5 + (M * cfg.topk > 1024)  # routed + dense launches
        run = PU.Run(tail, PU.to_cuda(act), cfg)
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()
    o = T.tail(act, w, cfg, tokens=tokens)
    PU.check_routing(run, o, cfg)
    return PU.check_stages(run, o, cfg, combine_buffer=not flags & B.KLT_FLAG_DETERMINISTIC)


def _small(**kw):
    base = dict(routed_fmt=FMT, I=256, E=8, topk=2, seed=81)
    base.update(kw)
    return configs.SMALL.with_(**base)


@pytest.mark.parametrize("M", [5, 40, 300])
def test_w4a4_small(M):
    _case(_small(), M)


def test_w4a4_several_tiles_in_every_dimension():
    _case(_small(H=768, L=512, I=512, Is=256, topk=3, seed=82), 150)


def test_w4a4_deterministic_combine():
    _case(_small(topk=3, seed=83), 40, flags=B.KLT_FLAG_DETERMINISTIC)


def test_w4a4_one_hot_and_zero_latent_rows():
    # a token whose latent row is all zero quantises to zero codes and zero scales; a
    # token routed with a huge logit margin sends all its weight to one expert
    cfg = _small(seed=84)
    M = 24
    w = inputs.make_weights(cfg)
    act = inputs.make_activations(cfg, M)
    act["z"][3] = 0
    act["logits"][5, 2] += 50.0
    tail = B.LatentMoETail(cfg, PU.to_cuda(w), max_tokens=M)
    try:
        run = PU.Run(tail, PU.to_cuda(act), cfg)
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()
    o = T.tail(act, w, cfg)
    PU.check_routing(run, o, cfg)
    PU.check_stages(run, o, cfg)
    assert not run.host("zq").numpy()[3].any() and not run.host("zsx").numpy()[3].any()


def test_w4a4_rejected_where_the_token_major_engine_is_not_available():
    for bad in (dict(H=384), dict(I=384)):  # H or I not a multiple of 256
        cfg = _small(**bad)
        w = PU.to_cuda(inputs.make_weights(cfg))
        with pytest.raises(B.KltError) as ei:
            B.LatentMoETail(cfg, w, max_tokens=8)
        assert ei.value.code == B.KLT_ERR_UNSUPPORTED


def test_w4a4_decode_m16_full_size():
    print("rel_fro", _case(configs.DECODE_M16_W4A4, 16))


@pytest.mark.slow
def test_w4a4_prefill_m8192_sampled_tokens():
    cfg = configs.PREFILL_M8192_W4A4
    rng = np.random.default_rng(6)
    tok = np.sort(rng.choice(cfg.M, 40, replace=False))
    tok[0], tok[-1] = 0, cfg.M - 1
    _case(cfg, cfg.M, tokens=tok)
