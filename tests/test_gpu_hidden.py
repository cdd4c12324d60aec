"""The step before the tail on the GPU (klt_forward_hidden) against the float64 oracle.

The library computes the latent input z = bf16(x W_lat^T) and the router logits
x W_gate^T from the hidden state, then runs the tail.  Checked, through the C ABI:
  * z against the oracle's correctly rounded bf16 values: 99 % equal; the rest within one
    bf16 step plus the fp32 accumulation error (16 fp32 units of the sum of |x_i w_i|);
  * the logits within the fp32 accumulation error of a 7168-term sum;
  * everything after the projection, bit for bit where the tail is (routing, permutation,
    latent codes) and within the output bar elsewhere, against the oracle run on the z
    and logits the GPU produced;
  * the output against the oracle run from x alone, on inputs whose top-k margins are far
    above the logits' error (so both sides route alike)."""
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


def _bf16_steps(got, ref):
    """Distance in bf16 steps (of the reference's binade) between bf16 values."""
    ref = np.asarray(ref, dtype=np.float64)
    ulp = np.where(ref == 0, 2.0 ** -133, 2.0 ** (np.floor(np.log2(np.abs(ref) + 1e-300)) - 7))
    return np.abs(np.asarray(got, dtype=np.float64) - ref) / ulp


def _run(cfg, M, force_bn=0, expect_tile=None):
    w = inputs.make_weights(cfg)
    w.update(inputs.make_projection_weights(cfg))
    act = inputs.make_activations(cfg, M)
    tail = B.LatentMoETail(cfg, PU.to_cuda(w), max_tokens=M)
    try:
        if expect_tile is not None:
            assert tail.gemm_tile(M) == expect_tile
        run = PU.Run(tail, PU.to_cuda(act), cfg, force_bn=force_bn, hidden=True)
        assert tail.status() == B.KLT_OK
    finally:
        tail.close()
    return w, act, run


def _check(cfg, w, act, run, tokens=None):
    z_o, lg_o = T.latent_inputs(act["x"], w["w_lat"], w["w_gate"])
    z_g = run.host("z").to(torch.float64).numpy()
    lg_g = run.host("logits").numpy().astype(np.float64)
    # the GPU sums in fp32: next to zero its error spans several of z's (tiny) bf16 steps,
    # so the bar is one bf16 step of z plus 16 fp32 units of the sum of |x_i w_i|
    S = np.abs(T.to_f64(act["x"])) @ np.abs(T.to_f64(w["w_lat"])).T
    steps = _bf16_steps(z_g, z_o)
    bound = 2.0 ** (np.floor(np.log2(np.abs(z_o) + 1e-300)) - 7) + 2.0 ** -20 * S
    bad = np.abs(z_g - z_o) > bound
    assert not bad.any(), f"{int(bad.sum())} z elements beyond the bound"
    assert (steps == 0).mean() >= 0.99, f"z exact in {(steps == 0).mean():.4%}"
    np.testing.assert_allclose(lg_g, lg_o, rtol=0, atol=2e-4)
    # everything after the projection, on the GPU's own z and logits
    act_g = {"x": act["x"], "z": run.host("z"), "logits": run.host("logits")}
    o = T.tail(act_g, w, cfg, tokens=tokens)
    PU.check_routing(run, o, cfg)
    PU.check_stages(run, o, cfg)
    # end to end from x: the oracle routes on its own float64 logits; both sides agree when
    # every token's k-th and (k+1)-th logits are further apart than the logits' error
    srt = -np.sort(-lg_o, axis=1)
    margin = srt[:, cfg.topk - 1] - srt[:, cfg.topk] if cfg.topk < cfg.E else np.inf
    act_o = {"x": act["x"], "z": torch.from_numpy(z_o).to(torch.bfloat16),
             "logits": torch.from_numpy(lg_o)}
    o2 = T.tail(act_o, w, cfg, tokens=tokens)
    tok = o2["tokens"]
    safe = np.ones(len(tok), dtype=bool) if np.isscalar(margin) else margin[tok] > 1e-3
    assert safe.mean() > 0.8
    PU.assert_output_close(run.host("out").float().numpy()[tok][safe].astype(np.float64),
                           o2["out"][safe])


@pytest.mark.parametrize("M,bn", [(5, 16), (40, 256)])  # feature-major / token-major tail
@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_hidden_small(M, bn, fmt):
    cfg = configs.SMALL.with_(E=8, topk=2, routed_fmt=fmt, seed=61)
    w, act, run = _run(cfg, M, expect_tile=bn)
    _check(cfg, w, act, run)


@pytest.mark.parametrize("fmt,M", [("mxfp8", 12), ("nvfp4_w4a4", 12), ("nvfp4_w4a4", 150)])
def test_hidden_block_scaled_formats(fmt, M):
    # the projection feeds the block-scaled routed formats the same way (their latent
    # quantisation happens in the routing kernel on the projected z)
    cfg = configs.SMALL.with_(E=8, topk=2, I=256, routed_fmt=fmt, seed=63)
    w, act, run = _run(cfg, M, expect_tile=256)
    _check(cfg, w, act, run)


def test_hidden_wider_shapes_and_gate_padding():
    # E = 40 gate rows padded with zero rows to a multiple of 128 after L = 384 latent rows
    cfg = configs.SMALL.with_(H=512, L=384, I=256, Is=256, E=40, topk=5, seed=62)
    w, act, run = _run(cfg, 23)
    _check(cfg, w, act, run)


def test_hidden_decode_m16_full_size():
    cfg = configs.DECODE_M16
    w, act, run = _run(cfg, 16, expect_tile=16)
    _check(cfg, w, act, run)


def test_hidden_rejected_without_projection_weights():
    cfg = configs.SMALL
    w = PU.to_cuda(inputs.make_weights(cfg))
    tail = B.LatentMoETail(cfg, w, max_tokens=4)
    try:
        x = torch.zeros((4, cfg.H), dtype=torch.bfloat16, device="cuda")
        out = torch.zeros((4, cfg.H), dtype=torch.bfloat16, device="cuda")
        assert B.klt_forward_hidden(tail.handle, x, 4, out) == B.KLT_ERR_UNSUPPORTED
    finally:
        tail.close()
