"""MLA attention over a paged FP8-e4m3 latent KV cache on one GB300 (sm_103a).

A thin ctypes binding over ``libmla.so`` (C ABI in ``include/mla.h``). The functions
carry the C names and only marshal arguments: torch CUDA tensors become device
pointers, the current torch stream becomes the ``cudaStream_t``. Every step of the
attention runs in the library's CUDA kernels; there is no other implementation, and
every entry point raises ImportError when the library is missing (the seeded workload
and accounting modules import without it).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_D = 576
MLA_DV = 512
MLA_OP_DECODE, MLA_OP_VERIFY, MLA_OP_PREFILL = 0, 1, 2
(MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA,
 MLA_ERR_TIMEOUT, MLA_ERR_BOUNDS) = range(7)
STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE",
          4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT", 6: "MLA_ERR_BOUNDS"}

# Every symbol include/mla.h declares.
EXPORTS = ("mla_workspace_size", "mla_decode", "mla_verify", "mla_prefill", "mla_merge_lse",
           "mla_read_status", "mla_status_string", "mla_last_launch_count",
           "mla_set_profile_events", "mla_decode_static_ws", "mla_cache_append",
           "mla_top_k_renorm_prob", "mla_verify_f32", "mla_prefill_mha",
           "mla_prefill_mha_workspace_size", "mla_test_stall_next_call",
           "mla_read_status_static", "mla_set_trace_buffer", "mla_verify_f32_shard",
           "mla_prefill_mha_bf16")


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}: "
                         f"{library().mla_status_string(status).decode()}")


class mla_kv_t(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_size", ctypes.c_int32), ("page_table", ctypes.c_void_p),
                ("page_table_stride", ctypes.c_int64), ("seq_lens", ctypes.c_void_p),
                ("kv_scale", ctypes.c_float)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmla.so not built at {LIB_PATH}: run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    KV = ctypes.POINTER(mla_kv_t)
    lib.mla_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.mla_workspace_size.restype = sz
    lib.mla_decode.argtypes = [KV, P, i32, i32, f32, P, P, P, sz, P]
    lib.mla_verify.argtypes = [KV, P, i32, i32, i32, f32, P, P, P, sz, P]
    lib.mla_verify_f32.argtypes = [KV, P, i32, i32, i32, f32, P, P, P, sz, P]
    lib.mla_verify_f32.restype = i32
    lib.mla_verify_f32_shard.argtypes = [KV, P, i32, i32, i32, f32, i32, P, P, P, sz, P]
    lib.mla_verify_f32_shard.restype = i32
    lib.mla_prefill_mha_workspace_size.argtypes = [i32, i32, i32]
    lib.mla_prefill_mha_workspace_size.restype = sz
    lib.mla_prefill_mha.argtypes = [KV, i32, P, i32, i32, P, f32, P, P, P, sz, P]
    lib.mla_prefill_mha.restype = i32
    lib.mla_prefill_mha_bf16.argtypes = [KV, i32, P, i32, i32, P, f32, P, P, P, sz, P]
    lib.mla_prefill_mha_bf16.restype = i32
    lib.mla_test_stall_next_call.argtypes = []
    lib.mla_test_stall_next_call.restype = None
    lib.mla_prefill.argtypes = [KV, P, i32, i32, f32, P, P, P, sz, P]
    lib.mla_merge_lse.argtypes = [P, P, i32, i64, P, P, P]
    lib.mla_read_status.argtypes = [P, sz, P]
    lib.mla_status_string.argtypes = [i32]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_last_launch_count.argtypes = []
    lib.mla_set_profile_events.argtypes = [P, P]
    lib.mla_set_profile_events.restype = None
    lib.mla_decode_static_ws.argtypes = [KV, P, i32, i32, f32, P, P, P]
    lib.mla_decode_static_ws.restype = i32
    lib.mla_read_status_static.argtypes = [P]
    lib.mla_read_status_static.restype = i32
    lib.mla_set_trace_buffer.argtypes = [P, sz]
    lib.mla_set_trace_buffer.restype = None
    lib.mla_cache_append.argtypes = [P, i64, i32, P, P, i64, f32, P, P]
    lib.mla_cache_append.restype = i32
    lib.mla_top_k_renorm_prob.argtypes = [P, P, i32, i32, P, i32, P]
    lib.mla_top_k_renorm_prob.restype = i32
    for name in ("mla_decode", "mla_verify", "mla_prefill", "mla_merge_lse", "mla_read_status",
                 "mla_last_launch_count"):
        getattr(lib, name).restype = i32
    return lib


_lib: Optional[ctypes.CDLL] = None


def library() -> ctypes.CDLL:
    """The loaded libmla.so (loaded on first use; raises ImportError if not built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


@dataclasses.dataclass
class KVCache:
    """Device-resident paged latent cache (see ``mla_kv_t`` in include/mla.h).
    pool uint8 [num_pages, page_size, 576]; page_table int32 [B, stride]; seq_lens int32 [B]."""

    pool: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    kv_scale: float

    def c_struct(self) -> mla_kv_t:
        for name in ("pool", "page_table", "seq_lens"):
            t = getattr(self, name)
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"KVCache.{name} must be a contiguous CUDA tensor")
        if self.pool.dtype != torch.uint8 or self.page_table.dtype != torch.int32 or \
                self.seq_lens.dtype != torch.int32:
            raise TypeError("KVCache dtypes: pool uint8, page_table int32, seq_lens int32")
        return mla_kv_t(self.pool.data_ptr(), self.pool.shape[0], self.pool.shape[1],
                        self.page_table.data_ptr(), self.page_table.shape[1],
                        self.seq_lens.data_ptr(), float(self.kv_scale))

    @staticmethod
    def from_inputs(inp, device="cuda") -> "KVCache":
        return KVCache(inp.pool.to(device), inp.page_table.to(device), inp.seq_lens.to(device),
                       inp.kv_scale)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MlaError(fn, status)


def mla_workspace_size(op: int, B: int, H: int, n_q: int, device: Optional[int] = None) -> int:
    if device is None:
        device = torch.cuda.current_device()
    return int(library().mla_workspace_size(op, B, H, n_q, device))


def workspace(op: int, B: int, H: int, n_q: int, device=None) -> torch.Tensor:
    """A zero-filled uint8 device buffer of the size mla_workspace_size() asks for."""
    n = mla_workspace_size(op, B, H, n_q, None if device is None else torch.device(device).index)
    if n == 0:
        raise ValueError("unsupported arguments for mla_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _q_check(q: torch.Tensor, ndim: int) -> None:
    if not q.is_cuda or q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != ndim or \
            q.shape[-1] != MLA_D:
        raise ValueError(f"q must be a contiguous CUDA bfloat16 tensor of rank {ndim} "
                         f"with last dimension {MLA_D}")


def mla_decode(kv: KVCache, q: torch.Tensor, sm_scale: float, out=None, lse=None, ws=None,
               stream=None):
    """q [B, H, 576] bf16 -> (out [B, H, 512] bf16, lse [B, H] fp32)."""
    _q_check(q, 3)
    B, H = q.shape[0], q.shape[1]
    out = torch.empty(B, H, MLA_DV, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty(B, H, dtype=torch.float32, device=q.device) if lse is None else lse
    ws = workspace(MLA_OP_DECODE, B, H, 1, q.device) if ws is None else ws
    c = kv.c_struct()
    _check("mla_decode", library().mla_decode(ctypes.byref(c), q.data_ptr(), B, H, sm_scale,
                                         out.data_ptr(), _ptr(lse), ws.data_ptr(), ws.numel(),
                                         _stream(stream)))
    return out, lse


def mla_verify(kv: KVCache, q: torch.Tensor, sm_scale: float, out=None, lse=None, ws=None,
               stream=None):
    """q [B, n_q, H, 576] bf16 -> (out [B, n_q, H, 512] bf16, lse [B, n_q, H] fp32)."""
    _q_check(q, 4)
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    out = torch.empty(B, n_q, H, MLA_DV, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty(B, n_q, H, dtype=torch.float32, device=q.device) if lse is None else lse
    ws = workspace(MLA_OP_VERIFY, B, H, n_q, q.device) if ws is None else ws
    c = kv.c_struct()
    _check("mla_verify", library().mla_verify(ctypes.byref(c), q.data_ptr(), B, n_q, H, sm_scale,
                                         out.data_ptr(), _ptr(lse), ws.data_ptr(), ws.numel(),
                                         _stream(stream)))
    return out, lse


def mla_prefill_mha(kv: KVCache, q: torch.Tensor, w_ukv: torch.Tensor, sm_scale: float,
                    L: Optional[int] = None, out=None, lse=None, ws=None, stream=None,
                    bf16: bool = False):
    """MHA-form causal prefill of sequence 0: q [T, H, 192] bf16, w_ukv [512, H, 256] bf16
    -> (out [T, H, 128] bf16, lse [T, H] fp32). L (cached positions incl. the T new ones)
    defaults to kv.seq_lens[0]. bf16=True calls mla_prefill_mha_bf16 (every tensor-core
    operand in bf16: faster, looser)."""
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[2] != 192 or not q.is_contiguous():
        raise ValueError("q must be a contiguous bfloat16 tensor [T, H, 192]")
    T, H = q.shape[0], q.shape[1]
    if w_ukv.dtype != torch.bfloat16 or tuple(w_ukv.shape) != (512, H, 256) or not w_ukv.is_contiguous():
        raise ValueError("w_ukv must be a contiguous bfloat16 tensor [512, H, 256]")
    if L is None:
        L = int(kv.seq_lens[0].item())
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty(T, H, dtype=torch.float32, device=q.device) if lse is None else lse
    if ws is None:
        n = int(library().mla_prefill_mha_workspace_size(L, H, q.device.index or 0))
        if n == 0:
            raise ValueError("no workspace size for these arguments")
        ws = torch.zeros(n, dtype=torch.uint8, device=q.device)
    c = kv.c_struct()
    name = "mla_prefill_mha_bf16" if bf16 else "mla_prefill_mha"
    _check(name, getattr(library(), name)(
        ctypes.byref(c), L, q.data_ptr(), T, H, w_ukv.data_ptr(), sm_scale, out.data_ptr(),
        _ptr(lse), ws.data_ptr(), ws.numel(), _stream(stream)))
    return out, lse


def mla_verify_f32(kv: KVCache, q: torch.Tensor, sm_scale: float, out=None, lse=None, ws=None,
                   stream=None, visible_shift: int = 0):
    """As mla_verify with a float32 output [B, n_q, H, 512], for results merged later.
    visible_shift > 0 moves every new position's causal limit that many keys later
    (mla_verify_f32_shard; n_q - 1 makes every key of the view visible to all of them)."""
    _q_check(q, 4)
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    out = torch.empty(B, n_q, H, MLA_DV, dtype=torch.float32, device=q.device) if out is None else out
    if out.dtype != torch.float32 or not out.is_contiguous() or out.shape != (B, n_q, H, MLA_DV):
        raise ValueError("out must be a contiguous float32 tensor [B, n_q, H, 512]")
    lse = torch.empty(B, n_q, H, dtype=torch.float32, device=q.device) if lse is None else lse
    ws = workspace(MLA_OP_VERIFY, B, H, n_q, q.device) if ws is None else ws
    c = kv.c_struct()
    if visible_shift == 0:
        _check("mla_verify_f32", library().mla_verify_f32(
            ctypes.byref(c), q.data_ptr(), B, n_q, H, sm_scale, out.data_ptr(), _ptr(lse),
            ws.data_ptr(), ws.numel(), _stream(stream)))
    else:
        _check("mla_verify_f32_shard", library().mla_verify_f32_shard(
            ctypes.byref(c), q.data_ptr(), B, n_q, H, sm_scale, int(visible_shift),
            out.data_ptr(), _ptr(lse), ws.data_ptr(), ws.numel(), _stream(stream)))
    return out, lse


def mla_prefill(kv: KVCache, q: torch.Tensor, sm_scale: float, out=None, lse=None, ws=None,
                stream=None):
    """q [T, H, 576] bf16 of one sequence -> (out [T, H, 512] bf16, lse [T, H] fp32)."""
    _q_check(q, 3)
    T, H = q.shape[0], q.shape[1]
    out = torch.empty(T, H, MLA_DV, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty(T, H, dtype=torch.float32, device=q.device) if lse is None else lse
    ws = workspace(MLA_OP_PREFILL, 1, H, T, q.device) if ws is None else ws
    c = kv.c_struct()
    _check("mla_prefill", library().mla_prefill(ctypes.byref(c), q.data_ptr(), T, H, sm_scale,
                                           out.data_ptr(), _ptr(lse), ws.data_ptr(), ws.numel(),
                                           _stream(stream)))
    return out, lse


def mla_merge_lse(part_out: torch.Tensor, part_lse: torch.Tensor, out=None, lse=None,
                  stream=None):
    """part_out [S, R, 512] fp32, part_lse [S, R] fp32 -> (out [R, 512] bf16, lse [R] fp32)."""
    if part_out.dtype != torch.float32 or part_lse.dtype != torch.float32 or \
            not part_out.is_contiguous() or not part_lse.is_contiguous():
        raise ValueError("partials must be contiguous float32 CUDA tensors")
    S, R = part_lse.shape
    out = torch.empty(R, MLA_DV, dtype=torch.bfloat16, device=part_out.device) if out is None else out
    lse = torch.empty(R, dtype=torch.float32, device=part_out.device) if lse is None else lse
    _check("mla_merge_lse", library().mla_merge_lse(part_out.data_ptr(), part_lse.data_ptr(), S, R,
                                               out.data_ptr(), _ptr(lse), _stream(stream)))
    return out, lse


def mla_cache_append(pool: torch.Tensor, x: torch.Tensor, slots: torch.Tensor, kv_scale: float,
                     status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write bf16 rows x [n, 576] into the uint8 pool [num_pages, page_size, 576] as e4m3
    codes of x / kv_scale at flat rows `slots` (int64 [n]; negative = skip). `status`, an
    int32 CUDA tensor of one element, receives MLA_ERR_BOUNDS for a slot past the pool."""
    if pool.dtype != torch.uint8 or pool.dim() != 3 or pool.shape[2] != MLA_D or not pool.is_contiguous():
        raise ValueError("pool must be a contiguous uint8 tensor [num_pages, page_size, 576]")
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != MLA_D or not x.is_contiguous():
        raise ValueError("x must be a contiguous bfloat16 tensor [n, 576]")
    if slots.dtype != torch.int64 or slots.dim() != 1 or slots.shape[0] != x.shape[0]:
        raise ValueError("slots must be an int64 tensor [n]")
    _check("mla_cache_append", library().mla_cache_append(
        pool.data_ptr(), pool.shape[0], pool.shape[1], x.data_ptr(), slots.data_ptr(),
        x.shape[0], float(kv_scale), None if status is None else status.data_ptr(),
        _stream(stream)))


def mla_top_k_renorm_prob(probs: torch.Tensor, top_k, out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """probs float32 [B, V] -> top-k renormalised copy; top_k an int (all rows) or an int32
    CUDA tensor [B]."""
    if probs.dtype != torch.float32 or probs.dim() != 2 or not probs.is_contiguous():
        raise ValueError("probs must be a contiguous float32 tensor [B, V]")
    B, V = probs.shape
    out = torch.empty_like(probs) if out is None else out
    if isinstance(top_k, torch.Tensor):
        if top_k.dtype != torch.int32 or top_k.shape != (B,):
            raise ValueError("top_k must be an int32 tensor [B]")
        kp, k = top_k.data_ptr(), 0
    else:
        kp, k = None, int(top_k)
    _check("mla_top_k_renorm_prob", library().mla_top_k_renorm_prob(
        probs.data_ptr(), out.data_ptr(), B, V, kp, k, _stream(stream)))
    return out


def mla_read_status(ws: torch.Tensor, stream=None) -> int:
    return int(library().mla_read_status(ws.data_ptr(), ws.numel(), _stream(stream)))


def mla_last_launch_count() -> int:
    return int(library().mla_last_launch_count())


def mla_set_profile_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event `start`/`stop` around the main attention kernel of the
    following calls on this thread (None, None switches it off)."""
    if (start is None) != (stop is None):
        raise ValueError("give both events or neither")
    library().mla_set_profile_events(None if start is None else start.cuda_event,
                                     None if stop is None else stop.cuda_event)
