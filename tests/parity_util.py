"""Helpers for the GPU parity tests: run the tail through the C ABI with every optional
output requested, and compare each stage with the float64 oracle."""
from __future__ import annotations

import ctypes
from typing import Dict, Optional

import numpy as np
import torch

from latent_moe_layer_route_gb300 import binding as B
from oracle import model as T
from oracle.codecs import e4m3_decode, unpack_e2m1

# Output bar of the tail (float): relative Frobenius error and per-element bound.
REL_FRO = 5e-3
ELEM_ABS_RMS = 0.03
ELEM_REL = 0.01


def to_cuda(d: Dict) -> Dict:
    return {k: (v.cuda() if hasattr(v, "cuda") else v) for k, v in d.items()}


class Run:
    """One forward with routing and stage outputs captured."""

    def __init__(self, tail: B.LatentMoETail, act: Dict, cfg, stall_after: int = 0,
                 timeout_ms: int = 0, force_bn: int = 0, hidden: bool = False):
        M = act["x"].shape[0]
        k, E, L, I, Is = cfg.topk, cfg.E, cfg.L, cfg.I, cfg.Is
        dev = "cuda"
        i32 = dict(dtype=torch.int32, device=dev)
        self.ids = torch.full((M, k), -7, **i32)
        self.w = torch.full((M, k), float("nan"), dtype=torch.float32, device=dev)
        self.cnt = torch.full((E,), -7, **i32)
        self.off = torch.full((E + 1,), -7, **i32)
        self.gidx = torch.full((M * k,), -7, **i32)
        self.slot = torch.full((M * k,), -7, **i32)
        self.pos = torch.full((M, k), -7, **i32)
        a4 = cfg.routed_fmt == "nvfp4_w4a4"  # codes packed two per byte
        self.zq = torch.zeros((M, L // 2 if a4 else L), dtype=torch.uint8, device=dev)
        self.zs = torch.zeros((M, L // 128), dtype=torch.float32, device=dev)
        self.aq = torch.zeros((M * k, I // 2 if a4 else I), dtype=torch.uint8, device=dev)
        self.as_ = torch.zeros((M * k, I // 128), dtype=torch.float32, device=dev)
        self.r = torch.zeros((M, L), dtype=torch.float32, device=dev)
        self.n = torch.zeros((M, L), dtype=torch.bfloat16, device=dev)
        self.a_s = torch.zeros((M, Is), dtype=torch.bfloat16, device=dev)
        self.out = torch.full((M, cfg.H), float("nan"), dtype=torch.bfloat16, device=dev)
        ro = B.KltRouting(*(t.data_ptr() for t in (self.ids, self.w, self.cnt, self.off,
                                                    self.gidx, self.slot, self.pos)))
        dbg = B.KltDebug()
        dbg.zq, dbg.zs, dbg.aq, dbg.as_ = (self.zq.data_ptr(), self.zs.data_ptr(),
                                           self.aq.data_ptr(), self.as_.data_ptr())
        dbg.r, dbg.n, dbg.a_s = self.r.data_ptr(), self.n.data_ptr(), self.a_s.data_ptr()
        dbg.stall_after_kblocks = stall_after
        dbg.timeout_ms = timeout_ms
        dbg.force_bn = force_bn
        if cfg.routed_fmt in ("mxfp8", "nvfp4_w4a4"):  # scale bytes of the latent input
            self.zsx = torch.zeros((M, L // (32 if cfg.routed_fmt == "mxfp8" else 16)),
                                   dtype=torch.uint8, device=dev)
            dbg.zsx = self.zsx.data_ptr()
        if hidden:  # latent input and logits computed from x by the library
            self.z = torch.zeros((M, L), dtype=torch.bfloat16, device=dev)
            self.logits = torch.full((M, E), float("nan"), dtype=torch.float32, device=dev)
            dbg.z, dbg.logits = self.z.data_ptr(), self.logits.data_ptr()
            tail.forward_hidden(act["x"], out=self.out, routing=ro, debug=dbg)
        else:
            tail.forward(act["x"], act["z"], act["logits"], out=self.out, routing=ro,
                         debug=dbg)
        torch.cuda.synchronize()

    def host(self, name):
        return getattr(self, name).cpu()


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def assert_output_close(got: np.ndarray, ref: np.ndarray, what: str = "out"):
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rf = rel_fro(got, ref)
    assert rf <= REL_FRO, f"{what}: relative Frobenius error {rf:.3e} > {REL_FRO}"
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = ELEM_ABS_RMS * rms + ELEM_REL * np.abs(ref)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements exceed "
                           f"0.03*rms+0.01*|ref| (worst {np.abs(got - ref).max():.3e})")
    return rf


def check_routing(run: Run, o: Dict, cfg, tokens: Optional[np.ndarray] = None):
    ids = run.host("ids").numpy()
    np.testing.assert_array_equal(ids, o["ids"])
    w = run.host("w").numpy().astype(np.float64)
    np.testing.assert_allclose(w, o["w"], rtol=1e-6, atol=1e-7)
    assert np.abs(w.sum(1) - 1.0).max() <= 1e-6
    np.testing.assert_array_equal(run.host("cnt").numpy(), o["cnt"])
    np.testing.assert_array_equal(run.host("off").numpy(), o["off"])
    np.testing.assert_array_equal(run.host("gidx").numpy(), o["gidx"])
    np.testing.assert_array_equal(run.host("slot").numpy(), o["slot"])
    np.testing.assert_array_equal(run.host("pos").numpy(), o["pos"])


def check_stages(run: Run, o: Dict, cfg, combine_buffer: bool = True):
    """Every stage for the oracle's selected tokens (o['tokens']).  `combine_buffer` False:
    the forward ran the fixed-order combine, which keeps no fp32 combine row (its sum is
    checked through the normalised latent and the output)."""
    tok = o["tokens"]
    a4 = cfg.routed_fmt == "nvfp4_w4a4"
    zq = run.host("zq").numpy()[tok]
    if a4:  # e2m1 codes, two per byte (even column in the low nibble)
        zq = unpack_e2m1(zq)
    np.testing.assert_array_equal(zq, o["zq"])
    pos = o["pos"][tok]
    aq = run.host("aq").numpy()[pos.reshape(-1)]
    if a4:
        aq = unpack_e2m1(aq)
    aq = aq.reshape(len(tok), cfg.topk, cfg.I)
    if cfg.routed_fmt in ("mxfp8", "nvfp4_w4a4"):
        # scale bytes of the latent input (UE8M0 or e4m3), exact; the routed activations'
        # scale bytes live in the tensor-core tiles only, so their codes are compared
        np.testing.assert_array_equal(run.host("zsx").numpy()[tok], o["zs"])
    else:
        np.testing.assert_array_equal(run.host("zs").numpy()[tok], o["zs"])
        # routed SwiGLU activations, compared through the decoded values per (token, choice)
        as_ = run.host("as_").numpy()[pos.reshape(-1)].reshape(len(tok), cfg.topk, -1)
        np.testing.assert_allclose(as_, o["as"], rtol=2e-3)
        deq_g = e4m3_decode(aq) * np.repeat(as_, 128, axis=-1)
        deq_o = e4m3_decode(o["aq"]) * np.repeat(o["as"], 128, axis=-1)
        assert rel_fro(deq_g, deq_o) < 2e-2
    code_diff = (aq != o["aq"]).mean()
    assert code_diff < 0.02, f"routed activation codes differ in {code_diff:.3%}"
    if combine_buffer:
        assert rel_fro(run.host("r").numpy()[tok].astype(np.float64), o["r"]) < REL_FRO
    a_s = run.host("a_s").float().numpy()[tok].astype(np.float64)
    assert rel_fro(a_s, o["a_s"]) < REL_FRO
    nn = run.host("n").float().numpy()[tok].astype(np.float64)
    assert rel_fro(nn, o["n"]) < REL_FRO
    return assert_output_close(run.host("out").float().numpy()[tok].astype(np.float64),
                               o["out"])
