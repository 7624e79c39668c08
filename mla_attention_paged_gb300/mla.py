"""Thin ctypes binding of libmla (include/mla.h).

Argument marshalling only: every step of the attention runs in the CUDA kernels behind the
C ABI.  PyTorch supplies device memory and the current stream.  If ``libmla.so`` has not
been built, importing this module raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE_TOO_SMALL = 3
MLA_ERR_CUDA = 4
MLA_ERR_TIMEOUT = 5
MLA_ERR_DEVICE_ARG = 6
MLA_KV_BF16 = 0
MLA_KV_E4M3 = 1
MLA_KV_INT8 = 2
MLA_KV_INT8_PAGE = 3

# Every function include/mla.h declares; each is given its C signature in _load().
EXPORTED = ["mla_decode_plan", "mla_decode", "mla_decode_partial", "mla_decode_combine", "mla_decode_noalloc",
            "mla_decode_int8_paged",
            "mla_prefill_varlen", "mla_prefill_paged", "mla_get_status", "mla_status_string", "mla_version", "mla_set_profile_events",
            "mla_profile_elapsed_ms", "mla_selftest_wait_timeout"]


class MlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what} failed: {status_string(code)} ({code})")


class DecodePlan(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_len", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("num_pages", ctypes.c_int64), ("num_sms", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("head_groups", ctypes.c_int32), ("chunk_tokens", ctypes.c_int32),
                ("max_splits", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("split_major", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmla.so is not built at {LIB_PATH}; run `python -m mla_attention_paged_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.mla_decode_plan.restype = i32
    lib.mla_decode_plan.argtypes = [i32, P, i32, i32, i32, i32, i64, i32, i32, ctypes.POINTER(DecodePlan)]
    lib.mla_decode.restype = i32
    lib.mla_decode.argtypes = [ctypes.POINTER(DecodePlan), P, P, P, P, i32, i32, f32, f32, P, P, P, sz, P]
    lib.mla_decode_partial.restype = i32
    lib.mla_decode_partial.argtypes = [ctypes.POINTER(DecodePlan), P, P, P, P, i32, i32, f32, f32, P, P, P, sz, P]
    lib.mla_decode_combine.restype = i32
    lib.mla_decode_noalloc.restype = i32
    lib.mla_decode_noalloc.argtypes = [ctypes.POINTER(DecodePlan), P, P, P, P, i32, i32, f32, f32, P, P, P]
    lib.mla_decode_combine.argtypes = [ctypes.POINTER(DecodePlan), P, i32, i32, P, P, P, sz, P]
    lib.mla_decode_int8_paged.restype = i32
    lib.mla_decode_int8_paged.argtypes = [ctypes.POINTER(DecodePlan), P, P, P, P, P, i32, i32, f32, f32, P, P, P,
                                          sz, P]
    lib.mla_prefill_varlen.restype = i32
    lib.mla_prefill_varlen.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, f32, P, P, P]
    lib.mla_prefill_paged.restype = i32
    lib.mla_prefill_paged.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, i32, i32, f32, P, P, P]
    lib.mla_get_status.restype = i32
    lib.mla_get_status.argtypes = [P]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [i32]
    lib.mla_version.restype = i32
    lib.mla_set_profile_events.restype = i32
    lib.mla_set_profile_events.argtypes = [P, P]
    lib.mla_profile_elapsed_ms.restype = i32
    lib.mla_selftest_wait_timeout.restype = i32
    lib.mla_selftest_wait_timeout.argtypes = [P]
    lib.mla_profile_elapsed_ms.argtypes = [P, P, ctypes.POINTER(ctypes.c_float)]
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.mla_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != MLA_OK:
        raise MlaError(code, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def decode_plan(seq_lens_host, q_len: int, num_heads: int, page_size: int, max_pages_per_seq: int,
                num_pages: int, kv_dtype: int = MLA_KV_BF16, num_sms: int = 0) -> DecodePlan:
    """Plan a decode launch from HOST sequence lengths (drafts included)."""
    lens = torch.as_tensor(seq_lens_host, dtype=torch.int32).cpu().contiguous()
    plan = DecodePlan()
    rc = lib.mla_decode_plan(int(lens.numel()), ctypes.c_void_p(lens.data_ptr()), int(q_len), int(num_heads),
                             int(page_size), int(max_pages_per_seq), int(num_pages), int(kv_dtype), int(num_sms),
                             ctypes.byref(plan))
    _check(rc, "mla_decode_plan")
    return plan


def workspace_for(plan: DecodePlan, device) -> torch.Tensor | None:
    """Allocate (with torch) a workspace of the size the plan asks for."""
    if plan.workspace_bytes == 0:
        return None
    return torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=device)


def decode(plan: DecodePlan, q: torch.Tensor, kv_pages: torch.Tensor, page_table: torch.Tensor,
           seq_lens: torch.Tensor, scale: float, kv_scale: float = 1.0, out=None, lse=None, workspace=None,
           stream=None):
    """mla_decode through the C ABI.  Returns (out [B,T,H,512] bf16, lse [B,T,H] fp32)."""
    B, T, H, D = q.shape
    if out is None:
        out = torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, H, dtype=torch.float32, device=q.device)
    if workspace is None and plan.workspace_bytes:
        workspace = workspace_for(plan, q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.mla_decode(ctypes.byref(plan), _ptr(q), _ptr(kv_pages), _ptr(page_table), _ptr(seq_lens), int(T),
                        int(H), float(scale), float(kv_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                        int(ws_bytes), _stream_handle(stream))
    _check(rc, "mla_decode")
    return out, lse


def decode_int8_paged(plan: DecodePlan, q: torch.Tensor, kv_pages: torch.Tensor, page_scales: torch.Tensor,
                      page_table: torch.Tensor, seq_lens: torch.Tensor, scale: float, kv_scale: float, out=None,
                      lse=None, workspace=None, stream=None):
    """mla_decode_int8_paged through the C ABI: an int8 pool with one fp32 scale per page
    (page_scales [num_pages] on the device).  Returns (out [B,T,H,512] bf16, lse [B,T,H] fp32)."""
    B, T, H, D = q.shape
    if out is None:
        out = torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, H, dtype=torch.float32, device=q.device)
    if workspace is None and plan.workspace_bytes:
        workspace = workspace_for(plan, q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.mla_decode_int8_paged(ctypes.byref(plan), _ptr(q), _ptr(kv_pages), _ptr(page_scales), _ptr(page_table),
                                   _ptr(seq_lens), int(T), int(H), float(scale), float(kv_scale), _ptr(out),
                                   _ptr(lse), _ptr(workspace), int(ws_bytes), _stream_handle(stream))
    _check(rc, "mla_decode_int8_paged")
    return out, lse


def decode_partial(plan: DecodePlan, q: torch.Tensor, kv_pages: torch.Tensor, page_table: torch.Tensor,
                   seq_lens: torch.Tensor, scale: float, kv_scale: float = 1.0, out=None, lse=None,
                   workspace=None, stream=None):
    """mla_decode_partial through the C ABI (stage 1 of decode): returns (out, lse, workspace);
    multi-split requests are finished by decode_combine with the same out/lse/workspace."""
    B, T, H, D = q.shape
    if out is None:
        out = torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, H, dtype=torch.float32, device=q.device)
    if workspace is None and plan.workspace_bytes:
        workspace = workspace_for(plan, q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.mla_decode_partial(ctypes.byref(plan), _ptr(q), _ptr(kv_pages), _ptr(page_table), _ptr(seq_lens),
                                int(T), int(H), float(scale), float(kv_scale), _ptr(out), _ptr(lse),
                                _ptr(workspace), int(ws_bytes), _stream_handle(stream))
    _check(rc, "mla_decode_partial")
    return out, lse, workspace


def decode_combine(plan: DecodePlan, seq_lens: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, workspace=None,
                   stream=None):
    """mla_decode_combine through the C ABI (stage 2 of decode): merges the split partials
    left in `workspace` by decode_partial into out/lse."""
    B, T, H, _ = out.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.mla_decode_combine(ctypes.byref(plan), _ptr(seq_lens), int(T), int(H), _ptr(out), _ptr(lse),
                                _ptr(workspace), int(ws_bytes), _stream_handle(stream))
    _check(rc, "mla_decode_combine")
    return out, lse


def decode_noalloc(plan: DecodePlan, q: torch.Tensor, kv_pages: torch.Tensor, page_table: torch.Tensor,
                   seq_lens: torch.Tensor, scale: float, kv_scale: float = 1.0, out=None, lse=None, stream=None):
    """mla_decode_noalloc through the C ABI: decode with the split-KV scratch in the
    library's fixed 32 MiB device buffer instead of a workspace.  Returns (out, lse)."""
    B, T, H, D = q.shape
    if out is None:
        out = torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, H, dtype=torch.float32, device=q.device)
    rc = lib.mla_decode_noalloc(ctypes.byref(plan), _ptr(q), _ptr(kv_pages), _ptr(page_table), _ptr(seq_lens),
                                int(T), int(H), float(scale), float(kv_scale), _ptr(out), _ptr(lse),
                                _stream_handle(stream))
    _check(rc, "mla_decode_noalloc")
    return out, lse


def prefill_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                   cu_seqlens_kv: torch.Tensor, prefix_lens: torch.Tensor, max_seqlen_q: int, scale: float,
                   out=None, lse=None, stream=None):
    """mla_prefill_varlen through the C ABI.  Returns (out [Nq,H,128] bf16, lse [Nq,H] fp32)."""
    Nq, H, _ = q.shape
    if out is None:
        out = torch.empty(Nq, H, v.shape[2], dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(Nq, H, dtype=torch.float32, device=q.device)
    rc = lib.mla_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(prefix_lens),
                                int(prefix_lens.numel()), int(H), int(max_seqlen_q), int(Nq), int(k.shape[0]),
                                float(scale), _ptr(out), _ptr(lse), _stream_handle(stream))
    _check(rc, "mla_prefill_varlen")
    return out, lse


def prefill_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, page_table: torch.Tensor,
                  cu_seqlens_q: torch.Tensor, kv_lens: torch.Tensor, max_seqlen_q: int, scale: float, out=None,
                  lse=None, stream=None):
    """mla_prefill_paged through the C ABI: the varlen prefill with K/V read through a page
    table from [num_pages, page_size, H, 192 | 128] pools.  Returns (out, lse)."""
    Nq, H, _ = q.shape
    num_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    if out is None:
        out = torch.empty(Nq, H, v_pages.shape[3], dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(Nq, H, dtype=torch.float32, device=q.device)
    rc = lib.mla_prefill_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(cu_seqlens_q),
                               _ptr(kv_lens), int(kv_lens.numel()), int(H), int(page_size), int(page_table.shape[1]),
                               int(num_pages), int(max_seqlen_q), int(Nq), float(scale), _ptr(out), _ptr(lse),
                               _stream_handle(stream))
    _check(rc, "mla_prefill_paged")
    return out, lse


def set_profile_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event pairs around the main kernel of later calls (this thread)."""
    lib.mla_set_profile_events(ctypes.c_void_p(start.cuda_event) if start is not None else None,
                               ctypes.c_void_p(stop.cuda_event) if stop is not None else None)


def profile_elapsed_ms(start, stop) -> float:
    """Milliseconds between two torch.cuda.Event objects recorded through the hook."""
    ms = ctypes.c_float()
    _check(lib.mla_profile_elapsed_ms(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event),
                                      ctypes.byref(ms)), "mla_profile_elapsed_ms")
    return ms.value


def selftest_wait_timeout(stream=None) -> None:
    """Enqueue the watchdog self-test kernel (its bounded wait must expire)."""
    _check(lib.mla_selftest_wait_timeout(_stream_handle(stream)), "mla_selftest_wait_timeout")


def get_status(stream=None) -> int:
    """Read and clear the device status word (synchronises the stream)."""
    return lib.mla_get_status(_stream_handle(stream))
