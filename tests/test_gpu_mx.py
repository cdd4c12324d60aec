"""The MXFP8 routed format (power-of-two scales per 32 K-elements, applied by the tensor
core's block-scaled MMA) against the float64 oracle, through the C ABI.

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
        run = PU.Run(tail, PU.to_cuda(act), cfg)
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()
    o = T.tail(act, w, cfg, tokens=tokens)
    PU.check_routing(run, o, cfg)
    return PU.check_stages(run, o, cfg, combine_buffer=not flags & B.KLT_FLAG_DETERMINISTIC)


@pytest.mark.parametrize("M", [5, 40, 300])
def test_mx_small(M):
    _case(configs.SMALL.with_(routed_fmt="mxfp8", E=8, topk=2, seed=71), M)


def test_mx_several_tiles_in_every_dimension():
    cfg = configs.SMALL.with_(routed_fmt="mxfp8", H=768, L=512, I=384, Is=256, E=8, topk=3,
                              seed=72)
    _case(cfg, 150)


def test_mx_deterministic_combine():
    _case(configs.SMALL.with_(routed_fmt="mxfp8", E=8, topk=3, seed=73), 40,
          flags=B.KLT_FLAG_DETERMINISTIC)


def test_mx_rejected_where_the_token_major_engine_is_not_available():
    cfg = configs.SMALL.with_(routed_fmt="mxfp8", H=384)  # H not a multiple of 256
    w = PU.to_cuda(inputs.make_weights(cfg))
    with pytest.raises(B.KltError) as ei:
        B.LatentMoETail(cfg, w, max_tokens=8)
    assert ei.value.code == B.KLT_ERR_UNSUPPORTED


def test_mx_decode_m16_full_size():
    print("rel_fro", _case(configs.DECODE_M16_MX, 16))


@pytest.mark.slow
def test_mx_prefill_m4096_sampled_tokens():
    cfg = configs.PREFILL_M4096_MX
    rng = np.random.default_rng(5)
    tok = np.sort(rng.choice(cfg.M, 40, replace=False))
    tok[0], tok[-1] = 0, cfg.M - 1
    _case(cfg, cfg.M, tokens=tok)
