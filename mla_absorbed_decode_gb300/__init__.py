"""GB300-native weight-absorbed MLA decode.

Python binding of ``libmla.so``, the C-ABI library declared in ``include/mla.h``.
The functions here only marshal arguments: every step of the path (schedule,
W_UK absorption, paged decode, LSE combine, W_UV un-absorption) runs in the
library's sm_103a kernels.  PyTorch supplies device memory and streams.
There is no fallback: if the library is not built, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MLAError", "lib", "library_path", "num_sm_parts", "metadata_size", "decode_metadata",
    "decode_workspace_size", "decode", "decode_sparse", "decode_fp8", "decode_sparse_fp8", "absorb_q", "unabsorb_o",
    "absorb_plan_max_batch", "absorb_q_plan",
    "bmm_fp8_workspace_size", "absorb_q_fp8", "absorb_q_fp8_plan", "unabsorb_o_fp8", "extend_workspace_size", "extend_chunked",
    "get_device_status",
    "schedule_params", "debug_withhold_first_load", "DecodeStep", "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE",
                4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT", 6: "MLA_ERR_DEVICE_BOUNDS"}

_c_int, _c_size, _c_float, _c_ll, _p = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_int64, ctypes.c_void_p
_SIGNATURES = {
    "mla_status_string": (ctypes.c_char_p, [_c_int]),
    "mla_num_sm_parts": (_c_int, [_c_int, _c_int, _c_int]),
    "mla_metadata_size": (_c_size, [_c_int, _c_int]),
    "mla_decode_metadata": (_c_int, [_p, _c_int, _c_int, _c_int, _c_int, _c_int, _p, _p]),
    "mla_schedule_params": (None, [ctypes.POINTER(_c_int), ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]),
    "mla_decode_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "mla_decode": (_c_int, [_p, _p, _c_ll, _p, _c_int, _p, _c_int, _c_int, _c_int, _c_float, _c_int,
                            _p, _c_int, _p, _c_size, _p, _p, _p]),
    "mla_decode_sparse": (_c_int, [_p, _p, _c_ll, _p, _c_int, _p, _p, _c_ll, _p, _c_int, _c_int, _c_int, _c_float,
                                   _c_int, _p, _c_int, _p, _c_size, _p, _p, _p]),
    "mla_decode_fp8": (_c_int, [_p, _p, _c_float, _c_ll, _p, _c_int, _p, _c_int, _c_int, _c_int, _c_float, _c_int,
                                _p, _c_int, _p, _c_size, _p, _p, _p]),
    "mla_decode_sparse_fp8": (_c_int, [_p, _p, _c_float, _c_ll, _p, _c_int, _p, _p, _c_ll, _p, _c_int, _c_int, _c_int,
                                       _c_float, _c_int, _p, _c_int, _p, _c_size, _p, _p, _p]),
    "mla_absorb_q": (_c_int, [_p, _c_ll, _p, _c_ll, _p, _p, _c_int, _c_int, _p]),
    "mla_absorb_q_rope": (_c_int, [_p, _c_ll, _p, _c_ll, _p, _c_float, _p, _p, _c_int, _c_int, _p]),
    "mla_absorb_plan_max_batch": (_c_int, []),
    "mla_absorb_q_plan": (_c_int, [_p, _c_ll, _p, _c_ll, _p, _c_float, _p, _p, _c_int, _c_int, _p, _c_int, _c_int, _p,
                                   _p]),
    "mla_unabsorb_o": (_c_int, [_p, _p, _p, _c_int, _c_int, _p]),
    "mla_bmm_fp8_workspace_size": (_c_size, []),
    "mla_absorb_q_fp8": (_c_int, [_p, _c_ll, _p, _c_ll, _p, _c_float, _p, _c_float, _p, _c_int, _c_int, _p, _c_size, _p]),
    "mla_absorb_q_fp8_plan": (_c_int, [_p, _c_ll, _p, _c_ll, _p, _c_float, _p, _c_float, _p, _c_int, _c_int, _p,
                                       _c_size, _p, _c_int, _c_int, _p, _p]),
    "mla_unabsorb_o_fp8": (_c_int, [_p, _p, _c_float, _p, _c_int, _c_int, _p, _c_size, _p]),
    "mla_extend_workspace_size": (_c_size, [_c_int, _c_int, _c_int]),
    "mla_extend_chunked": (_c_int, [_p, _p, _p, _p, _p, _c_ll, _p, _c_int, _c_int, _c_int, _c_float, _c_int, _p, _c_size,
                                    _p, _p, _p]),
    "mla_decode_noalloc": (_c_int, [_p, _p, _c_ll, _p, _c_int, _p, _c_int, _c_int, _c_int, _c_float, _c_int,
                                    _c_int, _p, _p, _p]),
    "mla_get_device_status": (_c_int, [_p]),
    "mla_debug_withhold_first_load": (None, [_c_int]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def lib() -> ctypes.CDLL:
    """Load libmla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it with "
                               "`python -m mla_absorbed_decode_gb300.build_lib`")
        handle = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int, what: str):
    if status != MLA_OK:
        raise MLAError(status, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def num_sm_parts(s_q: int, H: int, device: int | None = None) -> int:
    dev = torch.cuda.current_device() if device is None else device
    n = lib().mla_num_sm_parts(dev, s_q, H)
    if n <= 0:
        raise MLAError(-n if n < 0 else 4, "mla_num_sm_parts")
    return n


def metadata_size(B: int, parts: int) -> int:
    return lib().mla_metadata_size(B, parts)


def schedule_params() -> tuple[int, int, int]:
    """(set-up cost per segment, parts that saturate HBM, cost of an extra segment), in pages."""
    f, h, c = _c_int(), _c_int(), _c_int()
    lib().mla_schedule_params(ctypes.byref(f), ctypes.byref(h), ctypes.byref(c))
    return f.value, h.value, c.value


def decode_metadata(seqlens: torch.Tensor, s_q: int, H: int, causal: bool, parts: int,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Split-KV tile schedule for these sequence lengths (int32 tensor on the device)."""
    B = seqlens.numel()
    n_ints = metadata_size(B, parts) // 4
    if out is None:
        out = torch.empty(n_ints, dtype=torch.int32, device=seqlens.device)
    _check(lib().mla_decode_metadata(_ptr(seqlens), B, s_q, H, int(causal), parts, _ptr(out), _stream(stream)),
           "mla_decode_metadata")
    return out


def decode_workspace_size(B: int, s_q: int, H: int, parts: int) -> int:
    return lib().mla_decode_workspace_size(B, s_q, H, parts)


def decode(q, kv_cache, block_table, seqlens, softmax_scale: float, causal: bool, metadata, parts: int,
           workspace=None, out=None, lse=None, stream=None):
    """Absorbed MLA decode: returns (out [B,s_q,H,512] bf16, lse [B,s_q,H] fp32)."""
    B, s_q, H, _ = q.shape
    dev = q.device
    if out is None:
        out = torch.empty((B, s_q, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
    need = decode_workspace_size(B, s_q, H, parts)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(lib().mla_decode(_ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(block_table), block_table.shape[1],
                            _ptr(seqlens), B, s_q, H, float(softmax_scale), int(causal), _ptr(metadata), parts,
                            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
                            _stream(stream)), "mla_decode")
    return out, lse


def decode_sparse(q, kv_cache, block_table, seqlens, indices, topk_lens, softmax_scale: float, causal: bool, metadata,
                  parts: int, workspace=None, out=None, lse=None, stream=None):
    """Sparse (top-k) absorbed decode over indices[b, :topk_lens[b]] (int32 token positions);
    metadata from decode_metadata(topk_lens, ...).  Returns (out [B,s_q,H,512] bf16, lse [B,s_q,H] fp32)."""
    B, s_q, H, _ = q.shape
    dev = q.device
    if out is None:
        out = torch.empty((B, s_q, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, s_q, H, parts), dtype=torch.uint8, device=dev)
    _check(lib().mla_decode_sparse(_ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(block_table), block_table.shape[1],
                                   _ptr(seqlens), _ptr(indices), indices.stride(0), _ptr(topk_lens), B, s_q, H,
                                   float(softmax_scale), int(causal), _ptr(metadata), parts, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
                                   _stream(stream)), "mla_decode_sparse")
    return out, lse


def decode_fp8(q, kv_cache, kv_scale: float, block_table, seqlens, softmax_scale: float, causal: bool, metadata,
               parts: int, workspace=None, out=None, lse=None, stream=None):
    """Absorbed MLA decode over an FP8 cache: kv_cache [num_blocks,64,576] uint8 E4M3 codes (or a
    float8_e4m3fn tensor), cached value = code value * kv_scale.  Returns (out, lse) as decode."""
    B, s_q, H, _ = q.shape
    dev = q.device
    if kv_cache.element_size() != 1:
        raise TypeError("decode_fp8: kv_cache must hold one byte per value (E4M3 codes)")
    if out is None:
        out = torch.empty((B, s_q, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, s_q, H, parts), dtype=torch.uint8, device=dev)
    _check(lib().mla_decode_fp8(_ptr(q), _ptr(kv_cache), float(kv_scale), kv_cache.shape[0], _ptr(block_table),
                                block_table.shape[1], _ptr(seqlens), B, s_q, H, float(softmax_scale), int(causal),
                                _ptr(metadata), parts, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _ptr(out), _ptr(lse), _stream(stream)), "mla_decode_fp8")
    return out, lse


def decode_sparse_fp8(q, kv_cache, kv_scale: float, block_table, seqlens, indices, topk_lens, softmax_scale: float,
                      causal: bool, metadata, parts: int, workspace=None, out=None, lse=None, stream=None):
    """decode_sparse over an FP8 cache (E4M3 codes scaled by kv_scale, as in decode_fp8)."""
    B, s_q, H, _ = q.shape
    dev = q.device
    if kv_cache.element_size() != 1:
        raise TypeError("decode_sparse_fp8: kv_cache must hold one byte per value (E4M3 codes)")
    if out is None:
        out = torch.empty((B, s_q, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, s_q, H, parts), dtype=torch.uint8, device=dev)
    _check(lib().mla_decode_sparse_fp8(_ptr(q), _ptr(kv_cache), float(kv_scale), kv_cache.shape[0], _ptr(block_table),
                                       block_table.shape[1], _ptr(seqlens), _ptr(indices), indices.stride(0),
                                       _ptr(topk_lens), B, s_q, H, float(softmax_scale), int(causal), _ptr(metadata),
                                       parts, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
                                       _ptr(lse), _stream(stream)), "mla_decode_sparse_fp8")
    return out, lse


def absorb_q(q_nope: torch.Tensor, w_uk: torch.Tensor, q: torch.Tensor, q_pe: torch.Tensor | None = None,
             stream=None, positions: torch.Tensor | None = None, rope_theta: float = 10000.0) -> torch.Tensor:
    """q[n, h, 0:512] = q_nope[n, h, :] @ w_uk[h] and q[n, h, 512:576] = q_pe[n, h, :], RoPE-rotated
    by positions[n] (int32 [N]) when positions is given; q is [N, H, 576] (or [B, s_q, H, 576])."""
    N, H, _ = q_nope.shape
    pe_ptr, pe_stride = (0, 0) if q_pe is None else (_ptr(q_pe), q_pe.stride(0))
    if positions is None:
        _check(lib().mla_absorb_q(_ptr(q_nope), q_nope.stride(0), pe_ptr or None, pe_stride, _ptr(w_uk), _ptr(q), N,
                                  H, _stream(stream)), "mla_absorb_q")
    else:
        _check(lib().mla_absorb_q_rope(_ptr(q_nope), q_nope.stride(0), pe_ptr or None, pe_stride, _ptr(positions),
                                       float(rope_theta), _ptr(w_uk), _ptr(q), N, H, _stream(stream)),
               "mla_absorb_q_rope")
    return q


def absorb_plan_max_batch() -> int:
    return lib().mla_absorb_plan_max_batch()


def absorb_q_plan(q_nope: torch.Tensor, w_uk: torch.Tensor, q: torch.Tensor, seqlens: torch.Tensor, num_parts: int,
                  metadata: torch.Tensor, q_pe: torch.Tensor | None = None, positions: torch.Tensor | None = None,
                  rope_theta: float = 10000.0, stream=None) -> torch.Tensor:
    """absorb_q and decode_metadata(seqlens, ..., num_parts, out=metadata) in one launch
    (B = len(seqlens), s_q = N / B); returns q."""
    N, H, _ = q_nope.shape
    pe_ptr, pe_stride = (0, 0) if q_pe is None else (_ptr(q_pe), q_pe.stride(0))
    _check(lib().mla_absorb_q_plan(_ptr(q_nope), q_nope.stride(0), pe_ptr or None, pe_stride,
                                   _ptr(positions) if positions is not None else None, float(rope_theta), _ptr(w_uk),
                                   _ptr(q), N, H, _ptr(seqlens), seqlens.numel(), int(num_parts), _ptr(metadata),
                                   _stream(stream)), "mla_absorb_q_plan")
    return q


def unabsorb_o(o_lat: torch.Tensor, w_uv: torch.Tensor, o: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """o[n, h, :] = o_lat[n, h, :] @ w_uv[h]; o_lat is [N, H, 512] -> o [N, H, 128]."""
    N, H = o_lat.shape[0], o_lat.shape[1]
    if o is None:
        o = torch.empty((N, H, 128), dtype=torch.bfloat16, device=o_lat.device)
    _check(lib().mla_unabsorb_o(_ptr(o_lat), _ptr(w_uv), _ptr(o), N, H, _stream(stream)), "mla_unabsorb_o")
    return o


def bmm_fp8_workspace_size() -> int:
    return lib().mla_bmm_fp8_workspace_size()


def _fp8_workspace(dev, workspace):
    if workspace is None:
        workspace = torch.empty(bmm_fp8_workspace_size(), dtype=torch.uint8, device=dev)
    return workspace


def absorb_q_fp8(q_nope: torch.Tensor, w_uk_t: torch.Tensor, w_uk_scale: float, q: torch.Tensor,
                 q_pe: torch.Tensor | None = None, positions: torch.Tensor | None = None,
                 rope_theta: float = 10000.0, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q[n, h, 0:512] = bmm_fp8(input_to_float8(q_nope), W_UK)[n, h] with w_uk_t [H, 512, 128] E4M3
    codes (uint8 or float8_e4m3fn) and scale w_uk_scale; q[n, h, 512:576] = q_pe[n, h], RoPE-rotated
    by positions[n] when positions is given."""
    N, H, _ = q_nope.shape
    if w_uk_t.element_size() != 1:
        raise TypeError("absorb_q_fp8: w_uk_t must hold one E4M3 code per value")
    ws = _fp8_workspace(q_nope.device, workspace)
    pe_ptr, pe_stride = (0, 0) if q_pe is None else (_ptr(q_pe), q_pe.stride(0))
    _check(lib().mla_absorb_q_fp8(_ptr(q_nope), q_nope.stride(0), pe_ptr or None, pe_stride,
                                  None if positions is None else _ptr(positions), float(rope_theta), _ptr(w_uk_t),
                                  float(w_uk_scale), _ptr(q), N, H, _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "mla_absorb_q_fp8")
    return q


def absorb_q_fp8_plan(q_nope: torch.Tensor, w_uk_t: torch.Tensor, w_uk_scale: float, q: torch.Tensor,
                      seqlens: torch.Tensor, num_parts: int, metadata: torch.Tensor, q_pe: torch.Tensor | None = None,
                      positions: torch.Tensor | None = None, rope_theta: float = 10000.0,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """absorb_q_fp8 and decode_metadata(seqlens, ..., num_parts, out=metadata) in one pass
    (B = len(seqlens), s_q = N / B); returns q."""
    N, H, _ = q_nope.shape
    if w_uk_t.element_size() != 1:
        raise TypeError("absorb_q_fp8_plan: w_uk_t must hold one E4M3 code per value")
    ws = _fp8_workspace(q_nope.device, workspace)
    pe_ptr, pe_stride = (0, 0) if q_pe is None else (_ptr(q_pe), q_pe.stride(0))
    _check(lib().mla_absorb_q_fp8_plan(_ptr(q_nope), q_nope.stride(0), pe_ptr or None, pe_stride,
                                       None if positions is None else _ptr(positions), float(rope_theta),
                                       _ptr(w_uk_t), float(w_uk_scale), _ptr(q), N, H, _ptr(ws),
                                       ws.numel() * ws.element_size(), _ptr(seqlens), seqlens.numel(),
                                       int(num_parts), _ptr(metadata), _stream(stream)), "mla_absorb_q_fp8_plan")
    return q


def unabsorb_o_fp8(o_lat: torch.Tensor, w_uv_t: torch.Tensor, w_uv_scale: float, o: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """o[n, h, :] = bmm_fp8(input_to_float8(o_lat), W_UV)[n, h] with w_uv_t [H, 128, 512] E4M3 codes
    and scale w_uv_scale; o_lat is [N, H, 512] -> o [N, H, 128] bf16."""
    N, H = o_lat.shape[0], o_lat.shape[1]
    if w_uv_t.element_size() != 1:
        raise TypeError("unabsorb_o_fp8: w_uv_t must hold one E4M3 code per value")
    if o is None:
        o = torch.empty((N, H, 128), dtype=torch.bfloat16, device=o_lat.device)
    ws = _fp8_workspace(o_lat.device, workspace)
    _check(lib().mla_unabsorb_o_fp8(_ptr(o_lat), _ptr(w_uv_t), float(w_uv_scale), _ptr(o), N, H, _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)), "mla_unabsorb_o_fp8")
    return o


def extend_workspace_size(T: int, H: int, chunk_tokens: int) -> int:
    return lib().mla_extend_workspace_size(T, H, chunk_tokens)


def extend_chunked(q_nope: torch.Tensor, q_pe: torch.Tensor, w_uk: torch.Tensor, w_uv: torch.Tensor,
                   kv_cache: torch.Tensor, block_row: torch.Tensor, seqlen: int, softmax_scale: float,
                   chunk_tokens: int = 2048, workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, stream=None):
    """Chunked extend on the expanded path (MHA_CHUNKED_KV): the T new tokens (the last T of the
    request's seqlen cached tokens, causal) attend to the cache expanded chunk by chunk, merged by
    LSE.  q_nope [T,H,128], q_pe [T,H,64] (RoPE applied), w_uk [H,128,512], w_uv [H,512,128],
    block_row int32 [>= ceil(seqlen/64)].  Returns (out [T,H,128] bf16, lse [T,H] fp32)."""
    T, H, _ = q_nope.shape
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(extend_workspace_size(T, H, chunk_tokens), dtype=torch.uint8, device=dev)
    _check(lib().mla_extend_chunked(_ptr(q_nope), _ptr(q_pe), _ptr(w_uk), _ptr(w_uv), _ptr(kv_cache),
                                    kv_cache.shape[0], _ptr(block_row), int(seqlen), T, H, float(softmax_scale),
                                    int(chunk_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _ptr(out), _ptr(lse), _stream(stream)), "mla_extend_chunked")
    return out, lse


def get_device_status(stream=None) -> int:
    """Synchronize the stream; return and clear the kernels' device status word."""
    return lib().mla_get_device_status(_stream(stream))


def debug_withhold_first_load(enable: bool = True):
    lib().mla_debug_withhold_first_load(int(enable))


class DecodeStep:
    """One decode step of an MLA layer for a fixed batch shape: W_UK absorption,
    absorbed decode over the paged latent cache, LSE combine, W_UV un-absorption.

    Buffers (q, out, lse, o, metadata, workspace) are allocated once here, with
    torch, and reused; `run` launches only library kernels.  With kv_scale given, the
    cache passed to `run` / `capture` is an FP8 (E4M3) cache with that per-tensor scale.
    """

    def __init__(self, B: int, s_q: int, H: int, seqlens: torch.Tensor, causal: bool, softmax_scale: float,
                 parts: int | None = None, device="cuda", kv_scale: float | None = None):
        self.B, self.s_q, self.H = B, s_q, H
        self.causal, self.scale = causal, softmax_scale
        self.kv_scale = kv_scale
        self.parts = parts if parts is not None else num_sm_parts(s_q, H)
        dev = torch.device(device)
        self.q = torch.empty((B, s_q, H, 576), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((B, s_q, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
        self.o = torch.empty((B * s_q, H, 128), dtype=torch.bfloat16, device=dev)
        self.workspace = torch.empty(decode_workspace_size(B, s_q, H, self.parts), dtype=torch.uint8, device=dev)
        self.seqlens = seqlens
        self.metadata = decode_metadata(seqlens, s_q, H, causal, self.parts)
        self._plan_stream = torch.cuda.Stream(device=dev)

    def plan(self, stream=None):
        """Recompute the split schedule (after seqlens changed)."""
        decode_metadata(self.seqlens, self.s_q, self.H, self.causal, self.parts, out=self.metadata, stream=stream)

    def plan_beside(self, work):
        """plan() on a side stream while `work()` (stream work that does not read the
        metadata, such as the W_UK absorption) runs on the current stream; the current
        stream then waits for both.  The schedule sees everything issued before the call."""
        cur = torch.cuda.current_stream(self.q.device)
        self._plan_stream.wait_stream(cur)
        with torch.cuda.stream(self._plan_stream):
            self.plan()
        work()
        cur.wait_stream(self._plan_stream)

    def absorb_and_plan(self, q_nope, q_pe, w_uk, positions=None, rope_theta: float = 10000.0, stream=None):
        """The W_UK absorption and plan() in one launch (B <= absorb_plan_max_batch(); else the
        two calls, the schedule on a side stream beside the absorption)."""
        if self.B <= absorb_plan_max_batch():
            absorb_q_plan(q_nope, w_uk, self.q, self.seqlens, self.parts, self.metadata, q_pe=q_pe,
                          positions=positions, rope_theta=rope_theta, stream=stream)
        else:
            self.plan_beside(lambda: absorb_q(q_nope, w_uk, self.q, q_pe=q_pe, stream=stream, positions=positions,
                                              rope_theta=rope_theta))

    def _decode(self, kv_cache, block_table, stream=None):
        if self.kv_scale is None:
            decode(self.q, kv_cache, block_table, self.seqlens, self.scale, self.causal, self.metadata, self.parts,
                   workspace=self.workspace, out=self.out, lse=self.lse, stream=stream)
        else:
            decode_fp8(self.q, kv_cache, self.kv_scale, block_table, self.seqlens, self.scale, self.causal,
                       self.metadata, self.parts, workspace=self.workspace, out=self.out, lse=self.lse, stream=stream)

    def run(self, q_nope, q_pe, w_uk, w_uv, kv_cache, block_table, stream=None, positions=None,
            rope_theta: float = 10000.0):
        """q_nope [B*s_q,H,128], q_pe [B*s_q,H,64] -> o [B*s_q,H,128] (bf16); with positions
        (int32 [B*s_q]) q_pe is RoPE-rotated inside the absorption."""
        absorb_q(q_nope, w_uk, self.q, q_pe=q_pe, stream=stream, positions=positions, rope_theta=rope_theta)
        self._decode(kv_cache, block_table, stream=stream)
        unabsorb_o(self.out.view(self.B * self.s_q, self.H, 512), w_uv, o=self.o, stream=stream)
        return self.o

    def capture(self, q_nope, q_pe, w_uk, w_uv, kv_cache, block_table, plan=True, before=None, after=None,
                positions=None, rope_theta: float = 10000.0):
        """Record the step (plan() if `plan`, then run()) into a CUDA graph; `replay()` relaunches it
        with one host call.  `before` / `after` are optional callables whose stream work (for example
        copies of the step's inputs from pinned host buffers, or of its result back) is recorded in
        the same graph.  The graph holds the addresses of every buffer: refill them in place between
        replays.  The step runs once, uncaptured, first (one-time library set-up happens there)."""
        def absorb():
            absorb_q(q_nope, w_uk, self.q, q_pe=q_pe, positions=positions, rope_theta=rope_theta)

        def body():
            if before is not None:
                before()
            if plan:   # the schedule in the absorption's launch
                self.absorb_and_plan(q_nope, q_pe, w_uk, positions=positions, rope_theta=rope_theta)
            else:
                absorb()
            self._decode(kv_cache, block_table)
            unabsorb_o(self.out.view(self.B * self.s_q, self.H, 512), w_uv, o=self.o)
            if after is not None:
                after()
        side = torch.cuda.Stream(device=self.q.device)
        side.wait_stream(torch.cuda.current_stream(self.q.device))
        with torch.cuda.stream(side):
            body()
        torch.cuda.current_stream(self.q.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            body()
        self._graph = graph
        return graph

    def replay(self):
        """Relaunch the captured step on the current stream (see `capture`); returns o."""
        if getattr(self, "_graph", None) is None:
            raise RuntimeError("DecodeStep.replay() before capture()")
        self._graph.replay()
        return self.o
