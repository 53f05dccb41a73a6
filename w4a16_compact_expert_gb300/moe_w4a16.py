"""Thin ctypes binding of the C ABI in include/moe_w4a16.h.

Argument marshalling only: every step of the layer runs in the CUDA library.
PyTorch supplies device memory and the current stream.  The library is
loaded on first use; if it is missing (not built) the binding raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_w4a16.so")

OK, ERR_INVALID_ARG, ERR_CUDA, ERR_OOM, ERR_NOT_PACKED, ERR_NOT_RESIDENT, ERR_TIMEOUT, ERR_UNSUPPORTED = range(8)
STATUS_NAMES = ["OK", "ERR_INVALID_ARG", "ERR_CUDA", "ERR_OOM", "ERR_NOT_PACKED", "ERR_NOT_RESIDENT",
                "ERR_TIMEOUT", "ERR_UNSUPPORTED"]
RESIDUAL, PRENORM, FORCE_GEMV, FORCE_GEMM, UNFUSED, OFFLOAD = 1, 2, 4, 8, 16, 32

EXPORTED = ["moe_w4a16_create", "moe_w4a16_destroy", "moe_w4a16_pack_experts", "moe_w4a16_set_slot_table",
            "moe_w4a16_forward", "moe_w4a16_forward_host", "moe_w4a16_forward_host_async", "moe_w4a16_get_status", "moe_w4a16_last_error",
            "moe_w4a16_slot_bytes", "moe_w4a16_get_gemv_max_tokens", "moe_w4a16_set_gemv_max_tokens",
            "moe_w4a16_set_stage_events", "moe_w4a16_last_path", "moe_w4a16_route_noalloc",
            "moe_w4a16_cache_create", "moe_w4a16_cache_destroy", "moe_w4a16_cache_acquire",
            "moe_w4a16_cache_release", "moe_w4a16_cache_get_stats", "moe_w4a16_cache_slot_of",
            "moe_w4a16_cache_last_error", "moe_w4a16_cache_create_sim", "moe_w4a16_cache_sim_complete",
            "moe_w4a16_cache_sim_fail", "moe_w4a16_selftest_timeout", "moe_w4a16_offload_enable"]
PATH_NONE, PATH_DECODE_FUSED, PATH_DECODE, PATH_GEMM, PATH_OFFLOAD = 0, 1, 2, 3, 4
PATH_NAMES = {PATH_NONE: "none", PATH_DECODE_FUSED: "decode_fused", PATH_DECODE: "decode", PATH_GEMM: "gemm",
              PATH_OFFLOAD: "offload_qpacked"}


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("num_slots", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("device", ctypes.c_int32)]


class CacheConfig(ctypes.Structure):
    _fields_ = [("staging_experts", ctypes.c_int32), ("spare_slots", ctypes.c_int32), ("max_group", ctypes.c_int32)]


class CacheStats(ctypes.Structure):
    _fields_ = [("generation", ctypes.c_uint64), ("transactions", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("evictions", ctypes.c_uint64), ("h2d_bytes", ctypes.c_uint64),
                ("d2h_bytes", ctypes.c_uint64), ("lease_waits", ctypes.c_uint64), ("resident", ctypes.c_int32),
                ("free_spares", ctypes.c_int32), ("retiring", ctypes.c_int32), ("active_leases", ctypes.c_int32),
                ("faulted", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < 8 else status}: {msg}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load (once) and return the CUDA library; raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i32, u32, i64p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.POINTER(ctypes.c_int64)
    lib.moe_w4a16_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(vp)]
    lib.moe_w4a16_destroy.argtypes = [vp]
    lib.moe_w4a16_pack_experts.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.moe_w4a16_set_slot_table.argtypes = [vp, vp, vp]
    lib.moe_w4a16_forward.argtypes = [vp, vp, i32, vp, vp, u32, vp, vp, vp, vp, vp, vp]
    lib.moe_w4a16_forward_host.argtypes = [vp, vp, i32, vp, vp, u32, vp, vp]
    lib.moe_w4a16_forward_host_async.argtypes = [vp, vp, i32, vp, vp, u32, vp, vp]
    lib.moe_w4a16_get_status.argtypes = [vp, i64p]
    lib.moe_w4a16_last_error.argtypes = [vp]
    lib.moe_w4a16_last_error.restype = ctypes.c_char_p
    lib.moe_w4a16_slot_bytes.argtypes = [vp]
    lib.moe_w4a16_slot_bytes.restype = ctypes.c_size_t
    lib.moe_w4a16_get_gemv_max_tokens.argtypes = [vp]
    lib.moe_w4a16_get_gemv_max_tokens.restype = i32
    lib.moe_w4a16_set_gemv_max_tokens.argtypes = [vp, i32]
    lib.moe_w4a16_set_stage_events.argtypes = [vp, vp]
    lib.moe_w4a16_offload_enable.argtypes = [vp, i32]
    lib.moe_w4a16_last_path.argtypes = [vp, ctypes.POINTER(i32)]
    lib.moe_w4a16_last_path.restype = i32
    u64, u64p = ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64)
    lib.moe_w4a16_cache_create.argtypes = [vp, ctypes.POINTER(CacheConfig), vp, vp, vp, vp, vp, vp, vp, i32,
                                           ctypes.POINTER(vp)]
    lib.moe_w4a16_cache_create_sim.argtypes = [i32, i32, u64, ctypes.POINTER(CacheConfig), vp, i32,
                                               ctypes.POINTER(vp)]
    lib.moe_w4a16_cache_destroy.argtypes = [vp]
    lib.moe_w4a16_cache_acquire.argtypes = [vp, vp, i32, vp, u64p]
    lib.moe_w4a16_cache_release.argtypes = [vp, u64, vp]
    lib.moe_w4a16_cache_get_stats.argtypes = [vp, ctypes.POINTER(CacheStats)]
    lib.moe_w4a16_cache_slot_of.argtypes = [vp, i32]
    lib.moe_w4a16_cache_slot_of.restype = i32
    lib.moe_w4a16_cache_last_error.argtypes = [vp]
    lib.moe_w4a16_cache_last_error.restype = ctypes.c_char_p
    lib.moe_w4a16_cache_sim_complete.argtypes = [vp, u64]
    lib.moe_w4a16_cache_sim_fail.argtypes = [vp, i32]
    lib.moe_w4a16_selftest_timeout.argtypes = [vp, i32, ctypes.c_int64, vp]
    lib.moe_w4a16_route_noalloc.argtypes = [vp, i32, i32, i32, i32, vp, vp, u32, vp, vp, vp, vp, vp]
    _lib = lib
    return lib


def _ptr(a) -> Optional[int]:
    """Device or host address of a torch tensor / numpy array (None -> NULL)."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("numpy array must be C-contiguous")
        return a.ctypes.data
    if not a.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return a.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class MoELayer:
    """One W4A16 routed-expert MoE layer on one GPU (a library handle)."""

    def __init__(self, hidden: int, inter: int, num_experts: int, top_k: int, num_slots: Optional[int] = None,
                 max_tokens: int = 2048, device: int = 0):
        self.lib = load_library()
        self.cfg = Config(hidden, inter, num_experts, top_k, num_experts if num_slots is None else num_slots,
                          max_tokens, device)
        h = ctypes.c_void_p()
        st = self.lib.moe_w4a16_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if st != OK:
            raise MoEError(st, self.lib.moe_w4a16_last_error(None).decode())
        self.h = h
        self.device = device

    # -- helpers
    def _check(self, st: int):
        if st != OK:
            raise MoEError(st, self.lib.moe_w4a16_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.lib.moe_w4a16_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:   # noqa: BLE001 - interpreter shutdown
            pass

    @property
    def slot_bytes(self) -> int:
        return self.lib.moe_w4a16_slot_bytes(self.h)

    @property
    def gemv_max_tokens(self) -> int:
        return self.lib.moe_w4a16_get_gemv_max_tokens(self.h)

    @gemv_max_tokens.setter
    def gemv_max_tokens(self, v: int):
        self._check(self.lib.moe_w4a16_set_gemv_max_tokens(self.h, int(v)))

    def offload_enable(self, n_slots: int):
        """FP16 execution slots for the offload-qpacked comparison path (forward flag OFFLOAD)."""
        self._check(self.lib.moe_w4a16_offload_enable(self.h, int(n_slots)))

    def last_path(self):
        """(path, kernel launches) of the last forward: PATH_* and a count."""
        n = ctypes.c_int32(0)
        p = self.lib.moe_w4a16_last_path(self.h, ctypes.byref(n))
        return int(p), int(n.value)

    def selftest_timeout(self, which: int, limit_cycles: int, stream=None):
        """Enqueue the failure-detection self-test (a wait that runs out)."""
        self._check(self.lib.moe_w4a16_selftest_timeout(self.h, int(which), int(limit_cycles), _stream(stream)))

    # -- API
    def pack_experts(self, slot0: int, gate_q, gate_s, up_q, up_s, down_q, down_s, stream=None):
        """Canonical qpacked arrays (numpy or torch, host or device), leading axis = expert."""
        n = int(gate_q.shape[0])
        self._check(self.lib.moe_w4a16_pack_experts(self.h, slot0, n, _ptr(gate_q), _ptr(gate_s), _ptr(up_q),
                                                    _ptr(up_s), _ptr(down_q), _ptr(down_s), _stream(stream)))

    def set_slot_table(self, expert_to_slot, stream=None):
        t = np.ascontiguousarray(np.asarray(expert_to_slot, dtype=np.int32))
        self._check(self.lib.moe_w4a16_set_slot_table(self.h, t.ctypes.data, _stream(stream)))

    def forward(self, x, router_w, bias=None, flags: int = 0, out=None, debug: bool = False, stream=None):
        """x: cuda fp16 [T, H].  Returns out (and a dict of routing tensors if debug)."""
        import torch
        T = int(x.shape[0])
        if out is None:
            out = torch.empty_like(x)
        dbg = {}
        if debug:
            k, E = self.cfg.top_k, self.cfg.num_experts
            dev = x.device
            dbg = {"ids": torch.empty(T, k, dtype=torch.int32, device=dev),
                   "weights": torch.empty(T, k, dtype=torch.float32, device=dev),
                   "sorted_pairs": torch.empty(T * k, dtype=torch.int32, device=dev),
                   "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev)}
        self._check(self.lib.moe_w4a16_forward(
            self.h, _ptr(x), T, _ptr(router_w), _ptr(bias), flags, _ptr(out), _ptr(dbg.get("ids")),
            _ptr(dbg.get("weights")), _ptr(dbg.get("sorted_pairs")), _ptr(dbg.get("offsets")), _stream(stream)))
        return (out, dbg) if debug else out

    def forward_raw(self, x_ptr: int, T: int, router_w_ptr: int, bias_ptr, flags: int, out_ptr: int, stream_ptr):
        """Pointer-level forward (no torch objects), for timing loops."""
        return self.lib.moe_w4a16_forward(self.h, x_ptr, T, router_w_ptr, bias_ptr, flags, out_ptr,
                                          None, None, None, None, stream_ptr)

    def forward_host(self, x_host, router_w, bias=None, flags: int = 0, out_host=None, stream=None):
        """x_host: host fp16 [T, H] (numpy or pinned torch).  Synchronous."""
        T = int(x_host.shape[0])
        if out_host is None:
            out_host = np.empty_like(x_host)
        self._check(self.lib.moe_w4a16_forward_host(self.h, _ptr(x_host), T, _ptr(router_w), _ptr(bias), flags,
                                                    _ptr(out_host), _stream(stream)))
        return out_host

    def forward_host_async(self, x_host, router_w, out_host, bias=None, flags: int = 0, stream=None):
        """Enqueues H2D of x_host, the forward and D2H into out_host on `stream`
        and returns; out_host is valid after the stream synchronises.  Both
        host buffers should be pinned."""
        T = int(x_host.shape[0])
        self._check(self.lib.moe_w4a16_forward_host_async(self.h, _ptr(x_host), T, _ptr(router_w), _ptr(bias),
                                                          flags, _ptr(out_host), _stream(stream)))
        return out_host

    def set_stage_events(self, events):
        """events: 5 torch.cuda.Event(enable_timing=True) (or None to stop)."""
        if events is None:
            self._check(self.lib.moe_w4a16_set_stage_events(self.h, None))
            return
        arr = (ctypes.c_void_p * 5)(*[ev.cuda_event for ev in events])
        self._check(self.lib.moe_w4a16_set_stage_events(self.h, arr))

    def get_status(self):
        """(status code, miss count); synchronises the device and clears the word."""
        miss = ctypes.c_int64(0)
        st = self.lib.moe_w4a16_get_status(self.h, ctypes.byref(miss))
        return st, miss.value


def route_noalloc(x, router_w, bias, num_experts: int, top_k: int, flags: int = 0, stream=None):
    """Routing only, through moe_w4a16_route_noalloc (no handle, no device
    allocation inside the library).  Returns device tensors (ids [T, k],
    weights [T, k], sorted pairs [T*k], offsets [E+1])."""
    import torch
    lib = load_library()
    T, H = x.shape
    dev = x.device
    ids = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    w = torch.empty((T, top_k), dtype=torch.float32, device=dev)
    sp = torch.empty((T * top_k,), dtype=torch.int32, device=dev)
    off = torch.empty((num_experts + 1,), dtype=torch.int32, device=dev)
    st = lib.moe_w4a16_route_noalloc(_ptr(x), T, H, num_experts, top_k, _ptr(router_w), _ptr(bias), flags,
                                     _ptr(ids), _ptr(w), _ptr(sp), _ptr(off), _stream(stream))
    if st != OK:
        raise MoEError(st, lib.moe_w4a16_last_error(None).decode())
    return ids, w, sp, off


class ExpertCache:
    """The partial-residency miss path (moe_w4a16_cache_*): an immutable host
    backing of all experts, bounded pinned staging, spare slot rows,
    generation publication, leases and LRU discard eviction.

    ExpertCache(layer, backing, staging_experts, spare_slots, max_group, initial)
    attaches to a MoELayer; ExpertCache.sim(num_experts, num_slots, ...) is the
    host-only simulation (no GPU)."""

    def __init__(self, layer=None, backing=None, staging_experts=1, spare_slots=1, max_group=1, initial=(),
                 _sim=None):
        self.lib = load_library()
        self.cfg = CacheConfig(staging_experts, spare_slots, max_group)
        init = np.ascontiguousarray(np.asarray(list(initial), dtype=np.int32))
        h = ctypes.c_void_p()
        if _sim is not None:
            ne, ns, eb = _sim
            st = self.lib.moe_w4a16_cache_create_sim(ne, ns, eb, ctypes.byref(self.cfg),
                                                     init.ctypes.data if init.size else None, int(init.size),
                                                     ctypes.byref(h))
            self._keep = None
        else:
            arrays = [np.ascontiguousarray(a) for a in backing]
            self._keep = arrays   # the immutable backing must outlive the cache
            st = self.lib.moe_w4a16_cache_create(layer.h, ctypes.byref(self.cfg),
                                                 *[a.ctypes.data for a in arrays],
                                                 init.ctypes.data if init.size else None, int(init.size),
                                                 ctypes.byref(h))
        if st != OK:
            raise MoEError(st, self.lib.moe_w4a16_last_error(None).decode())
        self.c = h
        self.layer = layer
        self.is_sim = _sim is not None

    def _st(self, stream):
        return None if self.is_sim else _stream(stream)

    @classmethod
    def sim(cls, num_experts, num_slots, expert_bytes=1000, staging_experts=1, spare_slots=1, max_group=1,
            initial=()):
        return cls(None, None, staging_experts, spare_slots, max_group, initial,
                   _sim=(num_experts, num_slots, expert_bytes))

    def _check(self, st):
        if st != OK:
            raise MoEError(st, self.lib.moe_w4a16_cache_last_error(self.c).decode())

    def acquire(self, ids, stream=None) -> int:
        a = np.ascontiguousarray(np.asarray(list(ids), dtype=np.int32))
        lease = ctypes.c_uint64(0)
        self._check(self.lib.moe_w4a16_cache_acquire(self.c, a.ctypes.data if a.size else None, int(a.size),
                                                     self._st(stream), ctypes.byref(lease)))
        return lease.value

    def release(self, lease: int, stream=None):
        self._check(self.lib.moe_w4a16_cache_release(self.c, ctypes.c_uint64(lease), self._st(stream)))

    def stats(self) -> dict:
        s = CacheStats()
        self._check(self.lib.moe_w4a16_cache_get_stats(self.c, ctypes.byref(s)))
        return s.as_dict()

    def slot_of(self, expert: int) -> int:
        return self.lib.moe_w4a16_cache_slot_of(self.c, int(expert))

    def sim_complete(self, lease: int):
        self._check(self.lib.moe_w4a16_cache_sim_complete(self.c, ctypes.c_uint64(lease)))

    def sim_fail(self, where: int):
        self._check(self.lib.moe_w4a16_cache_sim_fail(self.c, int(where)))

    def close(self):
        if self.c:
            self._check(self.lib.moe_w4a16_cache_destroy(self.c))
            self.c = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
