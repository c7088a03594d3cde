"""Shared helpers of the parity tests: run the library, run the oracle, compare.

Tolerances (written here, used by every parity test):
* out: max |delta| <= 2e-2 absolute on bf16 outputs of unit-scale inputs.
  Inputs with x8 outlier rows are not unit-scale: the kernel feeds P to the
  tensor cores in bf16, whose rounding (at most 2^-9 relative per p_t) moves
  an output element by at most 2^-9 * A, A = sum_t p_t |v_t| (the attention-
  weighted magnitude of the values, from the oracle), and the bf16 output
  rounding adds at most 2^-9 |out| <= 2^-9 A.  There the bound is elementwise
  max(2e-2, 2^-7 * A), twice that arithmetic;
* out, relative: ||delta||_2 / ||ref||_2 <= 1e-2 (typical is ~3e-3: bf16
  rounding of P and of the output), which guards against the absolute bound
  being loose when |out| is small;
* lse: |delta| <= 1e-3 * max(1, |ref|); the chunked extend on the expanded path
  materializes its per-head keys in bf16 and adds, per row, the largest move that
  rounding can give a score it sees (expanded_score_allowance);
* integer schedule and indexing: bit-exact.
The FP8-cache decode is held to the same bounds against the oracle's decode over the
dequantized cache: inside the kernel q (scaled by a power of two) and P each travel as
a sum of two E4M3 terms -- exact for q's 8 significant bits, 2^-9 relative for P, the
size of the bf16 path's rounding of P -- which a CPU emulation of that arithmetic puts
at ~2e-3 relative L2, <= 5e-3 absolute and ~1e-7 relative on lse for unit-scale inputs
(the rebase threshold 2^6 with P offset 2^2 keeps small P values near E4M3's subnormals).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mla_absorbed_decode_gb300 import workloads as W

OUT_ABS = 2e-2
OUT_REL_ULP = 2.0 ** -7
OUT_REL_L2 = 1e-2
LSE_REL = 1e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_library(inp: dict, parts: int | None = None, device="cuda"):
    """Metadata + decode through the library; returns (out, lse, metadata) as CPU tensors."""
    import mla_absorbed_decode_gb300 as mla
    q = inp["q"].to(device)
    kv = inp["kv_cache"].to(device)
    bt = inp["block_table"].to(device)
    sl = inp["seqlens"].to(device)
    B, s_q, H, _ = q.shape
    P = parts if parts is not None else mla.num_sm_parts(s_q, H)
    meta = mla.decode_metadata(sl, s_q, H, inp["causal"], P)
    if "kv_scale" in inp:   # FP8 (E4M3) cache
        out, lse = mla.decode_fp8(q, kv, inp["kv_scale"], bt, sl, inp["softmax_scale"], inp["causal"], meta, P)
    else:
        out, lse = mla.decode(q, kv, bt, sl, inp["softmax_scale"], inp["causal"], meta, P)
    st = mla.get_device_status()
    assert st == 0, f"device status {st}"
    return out.cpu(), lse.cpu(), meta.cpu(), P


def oracle_decode(inp: dict, batches=None):
    """Oracle on all requests (or a subset); returns float64 arrays for those requests."""
    sel = list(range(inp["q"].shape[0])) if batches is None else list(batches)
    fp8 = "kv_scale" in inp
    kv = inp.get("_kv_np")
    if kv is None:   # an FP8 cache stays as its codes: the oracle dequantizes the rows it gathers
        kv = inp["kv_cache"].numpy() if fp8 else inp["kv_cache"].float().numpy()
        inp["_kv_np"] = kv
    q = to_np(inp["q"][sel])
    bt = inp["block_table"][sel].numpy()
    sl = inp["seqlens"][sel].numpy()
    if fp8:
        out, lse, out_abs = oracle.decode_fp8(q, kv, inp["kv_scale"], bt, sl, inp["softmax_scale"],
                                              causal=inp["causal"], with_abs=True)
    else:
        out, lse, out_abs = oracle.decode_absorbed(q, kv, bt, sl, inp["softmax_scale"], causal=inp["causal"],
                                                   with_abs=True)
    return out, lse, out_abs


def compare(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, ref_out: np.ndarray, ref_lse: np.ndarray,
            ref_abs: np.ndarray | None = None, what: str = "", lse_extra: np.ndarray | None = None,
            out_extra: np.ndarray | None = None):
    """ref_abs given (inputs with outliers): elementwise bound max(2e-2, 2^-7 * ref_abs).
    lse_extra (per row): an added allowance on lse for a path that rounds its keys to bf16
    before the scores (the expanded path; see expanded_score_allowance).  out_extra (per
    element): an added allowance on the output for the same reason (see
    expanded_output_allowance)."""
    o = to_np(out_gpu)
    lo = to_np(lse_gpu)
    assert o.shape == ref_out.shape, (o.shape, ref_out.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    d = np.abs(o - ref_out)
    bound = np.maximum(OUT_ABS, OUT_REL_ULP * ref_abs) if ref_abs is not None else OUT_ABS
    if out_extra is not None:
        bound = bound + out_extra
    worst = np.unravel_index(np.argmax(d - bound), d.shape)
    assert np.all(d <= bound), f"{what}: max|dout|={d.max():.4g} at {worst} (ref {ref_out[worst]:.4g})"
    nrm = np.linalg.norm(ref_out)
    if nrm > 0:
        rel = np.linalg.norm(o - ref_out) / nrm
        assert rel <= OUT_REL_L2, f"{what}: relative L2 error {rel:.3g}"
    both_inf = np.isneginf(lo) & np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lo), np.isneginf(ref_lse)), f"{what}: -inf lse mismatch"
    with np.errstate(invalid="ignore"):
        dl = np.where(both_inf, 0.0, np.abs(lo - ref_lse))
    lb = LSE_REL * np.maximum(1.0, np.abs(np.where(both_inf, 0.0, ref_lse)))
    if lse_extra is not None:
        lb = lb + lse_extra
    assert np.all(dl <= lb), f"{what}: max|dlse|={dl.max():.4g}"
    return float(d.max()), float(np.linalg.norm(o - ref_out) / max(nrm, 1e-30))


def make(w: W.Workload, seed=0, **kw):
    return W.make_inputs(w, seed=seed, **kw)


def expanded_output_allowance(score_allowance, ref_abs):
    """If every score of a row moves by at most d (score_allowance, per (query, head)), each
    softmax weight p_t moves by a factor within [e^-2d, e^2d] (numerator and normaliser each by
    at most e^d), so an output element sum_t p_t v_t moves by at most (e^2d - 1) sum_t p_t |v_t|
    = (e^2d - 1) * ref_abs.  Returns that bound per element (ref_abs [T, H, 128])."""
    return np.expm1(2.0 * np.asarray(score_allowance))[..., None] * np.asarray(ref_abs)


def expanded_score_allowance(q_nope, k_nope, softmax_scale, qpos):
    """The expanded path materializes each head's keys k = W_UK c in bf16: rounding moves a
    key value by at most 2^-9 of itself, so a score by at most
    2^-9 * softmax_scale * sum_d |q_d k_d|, and lse (a p-weighted mean of the scores' moves)
    by at most the largest of those over the keys a row sees.  Returns that bound per
    (query, head): q_nope [T, H, 128], k_nope [H, L, 128] (the oracle's expansion of the whole
    context), qpos [T] (each query sees keys at positions <= qpos)."""
    q = np.abs(np.asarray(q_nope, dtype=np.float64))
    k = np.abs(np.asarray(k_nope, dtype=np.float64))
    T, H, _ = q.shape
    out = np.zeros((T, H))
    for h in range(H):
        a = q[:, h, :] @ k[h].T                      # [T, L]
        for i in range(T):
            out[i, h] = a[i, : int(qpos[i]) + 1].max()
    return 2.0 ** -9 * softmax_scale * out
