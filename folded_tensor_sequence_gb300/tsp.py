"""Thin Python binding of libtsp's C ABI (argument marshalling only).

Every function has the name of the C entry point it calls and takes torch
tensors (device memory owned by the caller) in place of raw pointers.  All
computation happens in the CUDA kernels behind the C ABI; if the library is
missing this module raises instead of computing anything another way.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

TSP_OK, TSP_ERR_INVALID_ARG, TSP_ERR_UNSUPPORTED, TSP_ERR_CUDA, TSP_ERR_TIMEOUT, TSP_ERR_WORKSPACE = range(6)
TSP_F32, TSP_BF16 = 0, 1
(TSP_OP_ATTENTION_FWD, TSP_OP_GATED_MLP_FWD, TSP_OP_LAYER_FWD, TSP_OP_LAYER_BWD, TSP_OP_DECODE,
 TSP_OP_RANK_ATTENTION, TSP_OP_RANK_MLP) = range(7)
TSP_SHARD_ATTENTION, TSP_SHARD_MLP = 0, 1
TSP_STATIC_SCRATCH_BYTES = 32 << 20  # size of the static scratch array behind tsp_attention_fwd_static

EXPORTS = [
    "tsp_plan_create", "tsp_plan_destroy", "tsp_workspace_bytes", "tsp_saved_bytes", "tsp_status_string",
    "tsp_last_error_message", "tsp_pack_weights", "tsp_unpack_weights", "tsp_zigzag_permute",
    "tsp_zigzag_unpermute", "tsp_kv_gather", "tsp_attention_fwd", "tsp_gated_mlp_fwd", "tsp_layer_fwd",
    "tsp_layer_bwd", "tsp_sync_check", "tsp_debug_fail_next", "tsp_profile_enable", "tsp_profile_report",
    "tsp_attention_fwd_static", "tsp_debug_wait_timeout", "tsp_plan_create_gqa", "tsp_decode_step",
    "tsp_plan_set_deterministic", "tsp_plan_get_deterministic", "tsp_rank_shard_bytes", "tsp_rank_extract_shard",
    "tsp_rank_qkv", "tsp_rank_attention", "tsp_rank_mlp",
]


class TspError(RuntimeError):
    def __init__(self, status: int, what: str, message: str):
        super().__init__(f"{what}: status {status} ({message})")
        self.status = status


class _Weights(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_void_p), ("o", ctypes.c_void_p), ("gate_up", ctypes.c_void_p),
                ("down", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Loads libtsp.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libtsp is not built ({path} missing); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.tsp_plan_create.argtypes = [i32, i64, i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.tsp_plan_create_gqa.argtypes = [i32, i64, i32, i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.tsp_plan_destroy.argtypes = [vp]
        L.tsp_plan_destroy.restype = None
        L.tsp_plan_set_deterministic.argtypes = [vp, i32]
        L.tsp_plan_get_deterministic.argtypes = [vp]
        L.tsp_plan_get_deterministic.restype = i32
        L.tsp_workspace_bytes.argtypes = [vp, i32, i32]
        L.tsp_workspace_bytes.restype = sz
        L.tsp_saved_bytes.argtypes = [vp, i32]
        L.tsp_saved_bytes.restype = sz
        L.tsp_status_string.argtypes = [i32]
        L.tsp_status_string.restype = ctypes.c_char_p
        L.tsp_last_error_message.argtypes = []
        L.tsp_last_error_message.restype = ctypes.c_char_p
        L.tsp_pack_weights.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(_Weights), vp]
        L.tsp_unpack_weights.argtypes = [vp, ctypes.POINTER(_Weights), ctypes.POINTER(vp), vp]
        L.tsp_zigzag_permute.argtypes = [vp, i32, vp, vp, vp]
        L.tsp_zigzag_unpermute.argtypes = [vp, i32, vp, vp, vp]
        L.tsp_kv_gather.argtypes = [vp, i32, vp, vp, vp, vp, vp]
        L.tsp_attention_fwd.argtypes = [vp, i32, vp, ctypes.POINTER(_Weights), vp, vp, vp, sz, vp]
        L.tsp_gated_mlp_fwd.argtypes = [vp, i32, vp, ctypes.POINTER(_Weights), vp, vp, sz, vp]
        L.tsp_layer_fwd.argtypes = [vp, i32, vp, ctypes.POINTER(_Weights), vp, vp, vp, sz, vp]
        L.tsp_layer_bwd.argtypes = [vp, i32, vp, ctypes.POINTER(_Weights), vp, vp, vp, ctypes.POINTER(_Weights), vp,
                                    sz, vp]
        L.tsp_decode_step.argtypes = [vp, i32, i64, vp, ctypes.POINTER(_Weights), vp, vp, vp, vp, sz, vp]
        L.tsp_sync_check.argtypes = [vp]
        L.tsp_debug_fail_next.argtypes = [i32, i32]
        L.tsp_debug_fail_next.restype = None
        L.tsp_debug_wait_timeout.argtypes = [ctypes.c_uint, vp]
        L.tsp_attention_fwd_static.argtypes = [vp, i32, vp, ctypes.POINTER(_Weights), vp, vp, vp]
        L.tsp_rank_shard_bytes.argtypes = [vp, i32]
        L.tsp_rank_shard_bytes.restype = sz
        L.tsp_rank_extract_shard.argtypes = [vp, ctypes.POINTER(_Weights), i32, i32, vp, vp]
        L.tsp_rank_qkv.argtypes = [vp, i32, vp, vp, vp, vp, vp]
        L.tsp_rank_attention.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.tsp_rank_mlp.argtypes = [vp, i32, vp, vp, vp, vp, vp, sz, vp]
        L.tsp_profile_enable.argtypes = [i32]
        L.tsp_profile_enable.restype = None
        L.tsp_profile_report.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_int), i32]
        L.tsp_profile_report.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != TSP_OK:
        msg = lib().tsp_last_error_message().decode(errors="replace")
        raise TspError(status, what, msg)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        if not torch.cuda.is_available():
            return None  # host-only calls (validation) on a machine without a GPU
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- plan -------------------------------------------------------------------

class Plan:
    """Owns a tsp_plan*; mirrors its shape fields."""

    def __init__(self, handle: int, D, seq, hidden, heads, head_dim, ffn, dtype, kv_heads=None):
        self.handle = handle
        self.D, self.seq, self.hidden, self.heads, self.head_dim, self.ffn = D, seq, hidden, heads, head_dim, ffn
        self.kv_heads = heads if kv_heads is None else kv_heads
        self.dtype = dtype

    @property
    def kv_hidden(self) -> int:
        return self.kv_heads * self.head_dim

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == TSP_BF16 else torch.float32

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.tsp_plan_destroy(self.handle)
            self.handle = None


def tsp_plan_create(D: int, seq: int, hidden: int, heads: int, head_dim: int, ffn: int, dtype) -> Plan:
    if isinstance(dtype, str):
        dtype = TSP_BF16 if dtype == "bf16" else TSP_F32
    out = ctypes.c_void_p()
    _check(lib().tsp_plan_create(D, seq, hidden, heads, head_dim, ffn, dtype, ctypes.byref(out)), "tsp_plan_create")
    return Plan(out.value, D, seq, hidden, heads, head_dim, ffn, dtype)


def tsp_plan_create_gqa(D: int, seq: int, hidden: int, heads: int, kv_heads: int, head_dim: int, ffn: int,
                        dtype) -> Plan:
    if isinstance(dtype, str):
        dtype = TSP_BF16 if dtype == "bf16" else TSP_F32
    out = ctypes.c_void_p()
    _check(lib().tsp_plan_create_gqa(D, seq, hidden, heads, kv_heads, head_dim, ffn, dtype, ctypes.byref(out)),
           "tsp_plan_create_gqa")
    return Plan(out.value, D, seq, hidden, heads, head_dim, ffn, dtype, kv_heads)


def tsp_plan_set_deterministic(plan: Plan, deterministic: int) -> None:
    _check(lib().tsp_plan_set_deterministic(plan.handle, deterministic), "tsp_plan_set_deterministic")


def tsp_plan_get_deterministic(plan: Plan) -> int:
    return lib().tsp_plan_get_deterministic(plan.handle)


def plan_for(cfg) -> Plan:
    """Plan of a workload description (fields D, seq, hidden, heads, head_dim, ffn, dtype, kv_h)."""
    return tsp_plan_create_gqa(cfg.D, cfg.seq, cfg.hidden, cfg.heads, cfg.kv_h, cfg.head_dim, cfg.ffn, cfg.dtype)


def tsp_workspace_bytes(plan: Plan, batch: int, op: int) -> int:
    return lib().tsp_workspace_bytes(plan.handle, batch, op)


def tsp_saved_bytes(plan: Plan, batch: int) -> int:
    return lib().tsp_saved_bytes(plan.handle, batch)


def tsp_status_string(status: int) -> str:
    return lib().tsp_status_string(status).decode()


def tsp_last_error_message() -> str:
    return lib().tsp_last_error_message().decode(errors="replace")


def tsp_sync_check(stream=None) -> None:
    _check(lib().tsp_sync_check(_stream(stream)), "tsp_sync_check")


def tsp_debug_fail_next(status: int, count: int = 1) -> None:
    lib().tsp_debug_fail_next(status, count)


def tsp_debug_wait_timeout(timeout_us: int, stream=None) -> None:
    _check(lib().tsp_debug_wait_timeout(timeout_us, _stream(stream)), "tsp_debug_wait_timeout")


def tsp_profile_enable(on: bool) -> None:
    lib().tsp_profile_enable(1 if on else 0)


def tsp_profile_report(max_entries: int = 64):
    """[(step name, total ms, launches)] since the last report (waits for the GPU)."""
    names = (ctypes.c_char_p * max_entries)()
    ms = (ctypes.c_double * max_entries)()
    cnt = (ctypes.c_int * max_entries)()
    n = lib().tsp_profile_report(names, ms, cnt, max_entries)
    return [(names[i].decode(), ms[i], cnt[i]) for i in range(min(n, max_entries))]


# ---- weights -------------------------------------------------------------------

@dataclass
class PackedWeights:
    qkv: torch.Tensor
    o: torch.Tensor
    gate_up: torch.Tensor
    down: torch.Tensor

    def c(self) -> _Weights:
        return _Weights(self.qkv.data_ptr(), self.o.data_ptr(), self.gate_up.data_ptr(), self.down.data_ptr())


def empty_packed(plan: Plan, device="cuda") -> PackedWeights:
    h, F, dt = plan.hidden, plan.ffn, plan.torch_dtype
    return PackedWeights(
        qkv=torch.empty(h + 2 * plan.kv_hidden, h, dtype=dt, device=device),
        o=torch.empty(h, h, dtype=dt, device=device),
        gate_up=torch.empty(2 * F, h, dtype=dt, device=device),
        down=torch.empty(h, F, dtype=dt, device=device),
    )


CANONICAL = ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")


def tsp_pack_weights(plan: Plan, canonical: dict, packed: PackedWeights, stream=None) -> None:
    arr = (ctypes.c_void_p * 7)(*[canonical[k].data_ptr() for k in CANONICAL])
    w = packed.c()
    _check(lib().tsp_pack_weights(plan.handle, arr, ctypes.byref(w), _stream(stream)), "tsp_pack_weights")


def tsp_unpack_weights(plan: Plan, packed: PackedWeights, canonical: dict, stream=None) -> None:
    arr = (ctypes.c_void_p * 7)(*[canonical[k].data_ptr() for k in CANONICAL])
    w = packed.c()
    _check(lib().tsp_unpack_weights(plan.handle, ctypes.byref(w), arr, _stream(stream)), "tsp_unpack_weights")


# ---- layout --------------------------------------------------------------------

def tsp_zigzag_permute(plan: Plan, batch: int, x, xz, stream=None) -> None:
    _check(lib().tsp_zigzag_permute(plan.handle, batch, _ptr(x), _ptr(xz), _stream(stream)), "tsp_zigzag_permute")


def tsp_zigzag_unpermute(plan: Plan, batch: int, xz, x, stream=None) -> None:
    _check(lib().tsp_zigzag_unpermute(plan.handle, batch, _ptr(xz), _ptr(x), _stream(stream)),
           "tsp_zigzag_unpermute")


def tsp_kv_gather(plan: Plan, batch: int, kz, vz, k, v, stream=None) -> None:
    _check(lib().tsp_kv_gather(plan.handle, batch, _ptr(kz), _ptr(vz), _ptr(k), _ptr(v), _stream(stream)),
           "tsp_kv_gather")


# ---- layer -----------------------------------------------------------------------

def _ws_args(ws):
    if ws is None:
        return None, 0
    return ws.data_ptr(), ws.numel() * ws.element_size()


def tsp_attention_fwd(plan: Plan, batch: int, xz, weights: PackedWeights, a_out, lse, workspace, stream=None):
    w = weights.c()
    wp, wn = _ws_args(workspace)
    _check(lib().tsp_attention_fwd(plan.handle, batch, _ptr(xz), ctypes.byref(w), _ptr(a_out), _ptr(lse), wp, wn,
                                   _stream(stream)), "tsp_attention_fwd")


def tsp_attention_fwd_static(plan: Plan, batch: int, xz, weights: PackedWeights, a_out, lse, stream=None):
    """tsp_attention_fwd without a workspace: scratch comes from the library's static device array."""
    w = weights.c()
    _check(lib().tsp_attention_fwd_static(plan.handle, batch, _ptr(xz), ctypes.byref(w), _ptr(a_out), _ptr(lse),
                                          _stream(stream)), "tsp_attention_fwd_static")


def tsp_gated_mlp_fwd(plan: Plan, batch: int, hz, weights: PackedWeights, m_out, workspace, stream=None):
    w = weights.c()
    wp, wn = _ws_args(workspace)
    _check(lib().tsp_gated_mlp_fwd(plan.handle, batch, _ptr(hz), ctypes.byref(w), _ptr(m_out), wp, wn,
                                   _stream(stream)), "tsp_gated_mlp_fwd")


def tsp_layer_fwd(plan: Plan, batch: int, x, weights: PackedWeights, y, saved, workspace, stream=None):
    w = weights.c()
    wp, wn = _ws_args(workspace)
    _check(lib().tsp_layer_fwd(plan.handle, batch, _ptr(x), ctypes.byref(w), _ptr(y), _ptr(saved), wp, wn,
                               _stream(stream)), "tsp_layer_fwd")


def tsp_layer_bwd(plan: Plan, batch: int, x, weights: PackedWeights, saved, dy, dx, grads: PackedWeights, workspace,
                  stream=None):
    w = weights.c()
    g = grads.c()
    wp, wn = _ws_args(workspace)
    _check(lib().tsp_layer_bwd(plan.handle, batch, _ptr(x), ctypes.byref(w), _ptr(saved), _ptr(dy), _ptr(dx),
                               ctypes.byref(g), wp, wn, _stream(stream)), "tsp_layer_bwd")


def tsp_decode_step(plan: Plan, batch: int, pos: int, x_new, weights: PackedWeights, k_cache, v_cache, y_new,
                    workspace, stream=None):
    w = weights.c()
    wp, wn = _ws_args(workspace)
    _check(lib().tsp_decode_step(plan.handle, batch, pos, _ptr(x_new), ctypes.byref(w), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(y_new), wp, wn, _stream(stream)), "tsp_decode_step")


# ---- one rank of a multi-GPU layer ------------------------------------------------

def tsp_rank_shard_bytes(plan: Plan, kind: int) -> int:
    return lib().tsp_rank_shard_bytes(plan.handle, kind)


def tsp_rank_extract_shard(plan: Plan, packed: PackedWeights, shard: int, kind: int, out, stream=None) -> None:
    w = packed.c()
    _check(lib().tsp_rank_extract_shard(plan.handle, ctypes.byref(w), shard, kind, _ptr(out), _stream(stream)),
           "tsp_rank_extract_shard")


def tsp_rank_qkv(plan: Plan, batch: int, x_local, attn_shard, q_local, kv_local, stream=None) -> None:
    _check(lib().tsp_rank_qkv(plan.handle, batch, _ptr(x_local), _ptr(attn_shard), _ptr(q_local), _ptr(kv_local),
                              _stream(stream)), "tsp_rank_qkv")


def tsp_rank_attention(plan: Plan, rank: int, batch: int, q_local, kv_all, attn_shard, resid, h_out, workspace,
                       stream=None) -> None:
    wp, wn = _ws_args(workspace)
    _check(lib().tsp_rank_attention(plan.handle, rank, batch, _ptr(q_local), _ptr(kv_all), _ptr(attn_shard),
                                    _ptr(resid), _ptr(h_out), wp, wn, _stream(stream)), "tsp_rank_attention")


def tsp_rank_mlp(plan: Plan, batch: int, h_local, mlp_shard, resid, y_out, workspace, stream=None) -> None:
    wp, wn = _ws_args(workspace)
    _check(lib().tsp_rank_mlp(plan.handle, batch, _ptr(h_local), _ptr(mlp_shard), _ptr(resid), _ptr(y_out), wp, wn,
                              _stream(stream)), "tsp_rank_mlp")


def workspace(plan: Plan, batch: int, op: int, device="cuda") -> torch.Tensor:
    """A byte tensor of tsp_workspace_bytes(plan, batch, op) bytes (at least 16)."""
    n = max(16, tsp_workspace_bytes(plan, batch, op))
    return torch.empty(n, dtype=torch.uint8, device=device)
