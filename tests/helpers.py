"""Shared test helpers: seeded layers, margin-guarded tokens, GPU calls, comparisons."""

from __future__ import annotations

import numpy as np

from expert_ffn_decode_gb300 import synth
from oracle import moe_oracle as mo

# Selection margin: tokens whose ordered top-(k+1) selection scores (or whose
# kept/dropped group scores) come closer than this are redrawn, so fp32 (GPU)
# and fp64 (oracle) rounding cannot change the picks or their order.
MARGIN = 1e-4
# Output tolerance (relative L2 over a token's H outputs).
OUT_REL_L2 = 2e-3
# Routing-weight tolerance (relative, elementwise): the GPU forms logits with an
# fp32 dot of H terms, the oracle in fp64.
W_REL = 1e-5


def oracle_cfg(w: dict, flags: int = 0) -> mo.MoeConfig:
    return mo.MoeConfig(hidden=w["hidden"], n_experts=w["n_experts"], top_k=w["top_k"],
                        expert_ff=w["expert_ff"], shared_ff=w["shared_ff"], n_groups=w["n_groups"],
                        groups_used=w["groups_used"], qtype=w["qtype"], qtype_down=w.get("qtype_down", 0),
                        weights_scale=w["weights_scale"], norm_min=w.get("norm_min", mo.NORM_MIN),
                        flags=flags, swiglu_limit=w.get("swiglu_limit", 0.0),
                        swiglu_limit_shared=w.get("swiglu_limit_shared", 0.0),
                        rms_eps=w.get("rms_eps", 0.0))


def selection_gap(s: np.ndarray, w: dict) -> float:
    """Smallest gap that decides the ordered picks of one token (fp64 scores)."""
    k, G, Gu = w["top_k"], w["n_groups"], w["groups_used"]
    E = len(s)
    gaps = []
    allowed = np.ones(E, bool)
    if G > 1:
        per = E // G
        gs = np.array([np.sort(s[g * per:(g + 1) * per])[::-1][:2].sum() for g in range(G)])
        order = np.sort(gs)[::-1]
        if Gu < G:
            gaps.append(order[Gu - 1] - order[Gu])
        keep = np.argsort(-gs, kind="stable")[:Gu]
        allowed = np.isin(np.arange(E) // per, keep)
    top = np.sort(s[allowed])[::-1][:k + 1]
    gaps.extend(np.abs(np.diff(top)))
    return float(min(gaps)) if gaps else np.inf


def margin_tokens(layer: dict, w: dict, n: int, seed: int, stream: int = 1, norm=None, scale: float = 1.0,
                  transform=None):
    """n tokens from the seeded stream (times `scale`, then through `transform` if given),
    skipping draws within MARGIN of a tie; with a prologue norm vector the routing is that
    of the normalised token."""
    cfg = oracle_cfg(w)
    it = synth.token_stream(seed, w["hidden"], stream)
    out, redraws = [], 0
    while len(out) < n:
        x = (next(it) * np.float32(scale)).astype(np.float32)
        if transform is not None:
            x = transform(x)
        xr = x if norm is None else mo.rms_norm(x, norm, cfg.rms_eps)
        _, _, s = mo.route(xr, layer["router_w"], layer["bias"], cfg)
        if selection_gap(s[0], w) >= MARGIN:
            out.append(x)
        else:
            redraws += 1
        if redraws > 50 * (n + 1):
            raise RuntimeError("margin guard keeps rejecting tokens")
    return np.stack(out) if n else np.zeros((0, w["hidden"]), np.float32), redraws


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


# ---------------------------------------------------------------------------
# GPU side (imports torch lazily)
# ---------------------------------------------------------------------------

class GpuLayer:
    """A layer's bytes on the device plus the calls that run it."""

    def __init__(self, layer: dict, w: dict, device="cuda:0"):
        import torch
        self.torch = torch
        self.w = w
        self.dev = torch.device(device)
        t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)
        self.router_w = t(layer["router_w"])
        self.bias = t(layer["bias"])
        self.experts = t(layer["expert_blocks"])
        self.shared = t(layer["shared_blocks"])

    def run(self, x: np.ndarray, flags: int = 0, out_init=None, stream=None, workspace=None,
            want_topk=True):
        import expert_ffn_decode_gb300 as ffn
        torch = self.torch
        T, H = x.shape
        cfg = ffn.make_cfg(**{**self.w, "n_tokens": T, "flags": flags})
        xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(self.dev)
        out = (torch.from_numpy(np.ascontiguousarray(out_init, np.float32)).to(self.dev)
               if out_init is not None else torch.full((T, H), float("nan"), device=self.dev))
        ids = torch.full((T, self.w["top_k"]), -1, dtype=torch.int32, device=self.dev) if want_topk else None
        wts = torch.full((T, self.w["top_k"]), float("nan"), device=self.dev) if want_topk else None
        nbytes = ffn.moe_workspace_size(cfg)
        assert nbytes > 0, ffn.moe_last_error() if nbytes == 0 else ""
        ws = workspace if workspace is not None else torch.zeros(nbytes, dtype=torch.uint8, device=self.dev)
        st = stream if stream is not None else torch.cuda.current_stream(self.dev)
        rc = ffn.moe_ffn_forward_ex(xd, self.router_w, self.bias, self.experts, self.shared, cfg, out,
                                    ws, ws.numel(), st, ids, wts)
        ffn.check(rc)
        ffn.check(ffn.moe_workspace_status(ws, st))
        return (out.cpu().numpy(), ids.cpu().numpy() if want_topk else None,
                wts.cpu().numpy() if want_topk else None)


def compare(out, ids, wts, ref_out, ref_ids, ref_w, label=""):
    assert np.array_equal(ids, ref_ids), f"{label}: picks differ\n{ids}\n{ref_ids}"
    assert np.all(np.isfinite(wts)), label
    werr = np.max(np.abs(wts - ref_w) / np.maximum(np.abs(ref_w), 1e-30))
    assert werr <= W_REL, f"{label}: weight rel err {werr}"
    for t in range(out.shape[0]):
        e = rel_l2(out[t], ref_out[t])
        assert e <= OUT_REL_L2, f"{label}: token {t} rel-L2 {e}"
    return max(rel_l2(out[t], ref_out[t]) for t in range(out.shape[0])) if out.shape[0] else 0.0
