"""Python binding of libkvs (the C ABI declared in include/kvs.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  If the compiled
library is missing, importing the binding's functions raises: there is no
fallback.

Two layers:
  * ``kvs_*`` functions with the C names, taking raw pointers / handles;
  * ``Context``: owns torch-allocated device buffers for one pool and calls
    the same functions with tensors.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_build" / "libkvs.so"

KVS_OK, KVS_EINVAL, KVS_ENOMEM, KVS_ECUDA, KVS_ENOTFOUND, KVS_EEXIST, KVS_ETRUNC, \
    KVS_ETIMEOUT, KVS_EDEVICE = range(9)
STATUS_NAMES = ["OK", "EINVAL", "ENOMEM", "ECUDA", "ENOTFOUND", "EEXIST", "ETRUNC",
                "ETIMEOUT", "EDEVICE"]
KVS_SELECT_THRESH, KVS_SELECT_LOWFRAC = 0, 1
KVS_SELECT_LRFU = 2
KVS_KV_BF16, KVS_KV_FP8_E4M3, KVS_KV_KIVI2 = 0, 1, 2
KVS_KIVI_GROUP_TOKENS, KVS_KIVI_RESIDUAL = 32, 128
KVS_GATHER_DEMOTE, KVS_GATHER_MIRROR, KVS_GATHER_ASYNC = 1, 2, 4
KVS_MAX_CALL_SEQS = 256
KVS_PREFETCH_MAX = 4096
BLOCK_TOKENS = 16

c_u32, c_u64, c_i32, c_i64, c_dbl, c_sz, c_vp = (
    ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
    ctypes.c_size_t, ctypes.c_void_p)


class kvs_config(ctypes.Structure):
    _fields_ = [("num_layers", c_u32), ("num_q_heads", c_u32), ("num_kv_heads", c_u32),
                ("head_dim", c_u32), ("block_tokens", c_u32), ("pool_blocks", c_u32),
                ("max_seqs", c_u32), ("max_blocks_per_seq", c_u32), ("max_call_blocks", c_u32),
                ("staging_pages", c_u32), ("alpha", c_dbl), ("recency_window", c_u32),
                ("kv_dtype", c_u32), ("w_recency", c_dbl), ("w_ema", c_dbl), ("w_anchor", c_dbl),
                ("cut_lo", c_dbl), ("cut_hi", c_dbl), ("pool_seed", c_u64),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float), ("kivi_groups", c_u32),
                ("reserved1", c_u32)]


class kvs_sizes(ctypes.Structure):
    _fields_ = [("page_bytes", c_sz), ("pool_bytes", c_sz), ("table_bytes", c_sz),
                ("records_bytes", c_sz), ("mass_bytes", c_sz), ("workspace_bytes", c_sz),
                ("staging_bytes", c_sz), ("group_page_bytes", c_sz), ("group_pool_bytes", c_sz)]


class kvs_buffers(ctypes.Structure):
    _fields_ = [("pool", c_vp), ("block_table", c_vp), ("records", c_vp), ("mass", c_vp),
                ("workspace", c_vp), ("staging", c_vp), ("group_pool", c_vp)]


class kvs_key(ctypes.Structure):
    _fields_ = [("seq_id", c_u64), ("block_idx", c_u64)]


class kvs_gather_args(ctypes.Structure):
    _fields_ = [("mode", c_i32), ("flags", c_u32), ("frac", c_dbl), ("host_dst", c_vp),
                ("host_dst_bytes", c_sz), ("ids_dev", c_vp), ("slot_dev", c_vp),
                ("ids_capacity", c_u32), ("reserved0", c_u32), ("stream", c_vp),
                ("side_stream", c_vp)]


class kvs_gather_result(ctypes.Structure):
    _fields_ = [("n_selected", c_u32), ("n_pages", c_u32), ("n_staged", c_u32),
                ("n_demoted", c_u32), ("bytes_to_host", c_u64)]


# The 64-byte record of include/kvs.h (kvs_record), as a numpy dtype.
RECORD_DTYPE = np.dtype({
    "names": ["seq_id", "block_idx", "score", "last_touch", "count", "tier", "flags", "pad0",
              "prio", "mass", "reserved", "lrfu"],
    "formats": ["<u8", "<u8", "<f8", "<u8", "<u4", "u1", "u1", "<u2", "<f8", "<f4", ("u1", 4), "<f8"],
    "offsets": [0, 8, 16, 24, 32, 36, 37, 38, 40, 48, 52, 56],
    "itemsize": 64,
})

_SIGS = {
    "kvs_required_sizes": (ctypes.c_int, [ctypes.POINTER(kvs_config), ctypes.POINTER(kvs_sizes)]),
    "kvs_create": (ctypes.c_int, [ctypes.POINTER(kvs_config), ctypes.POINTER(kvs_buffers),
                                  ctypes.POINTER(c_vp)]),
    "kvs_destroy": (None, [c_vp]),
    "kvs_last_error": (ctypes.c_char_p, [c_vp]),
    "kvs_seq_add": (ctypes.c_int, [c_vp, c_u64, c_i64, c_u32, c_vp]),
    "kvs_seq_remove": (ctypes.c_int, [c_vp, c_u64, c_vp]),
    "kvs_append_tokens": (ctypes.c_int, [c_vp, c_u64, c_u32, c_vp, c_vp, c_vp]),
    "kvs_append_token": (ctypes.c_int, [c_vp, c_u64, c_vp, c_vp, c_vp]),
    "kvs_append_step": (ctypes.c_int, [c_vp, ctypes.POINTER(c_u64), c_u32, c_vp, c_vp, c_vp]),
    "kvs_decode_step": (ctypes.c_int, [c_vp, ctypes.POINTER(c_u64), c_u32, c_vp, c_vp, c_vp]),
    "kvs_decode_score_step": (ctypes.c_int, [c_vp, ctypes.POINTER(c_u64), c_u32, c_vp, c_vp, c_vp]),
    "kvs_score_update": (ctypes.c_int, [c_vp, c_vp]),
    "kvs_set_alpha": (ctypes.c_int, [c_vp, c_dbl]),
    "kvs_select_and_gather": (ctypes.c_int, [c_vp, ctypes.POINTER(kvs_gather_args),
                                             ctypes.POINTER(kvs_gather_result)]),
    "kvs_gather_counts": (ctypes.c_int, [c_vp, ctypes.POINTER(kvs_gather_result)]),
    "kvs_readmit": (ctypes.c_int, [c_vp, ctypes.POINTER(kvs_key), c_u32, c_vp, c_sz, c_vp]),
    "kvs_prefetch_plan": (ctypes.c_int, [c_vp, c_u32, ctypes.POINTER(kvs_key), ctypes.POINTER(c_dbl),
                                         ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(c_u32), c_vp]),
    "kvs_prefetch": (ctypes.c_int, [c_vp, c_u32, c_vp, c_sz, ctypes.POINTER(kvs_key), ctypes.POINTER(c_dbl),
                                    ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(c_u32), c_vp]),
    "kvs_debug_set_mass": (ctypes.c_int, [c_vp, ctypes.POINTER(c_u64), c_u32, c_vp, c_vp]),
    "kvs_debug_advance": (ctypes.c_int, [c_vp, c_u64]),
    "kvs_export_records": (ctypes.c_int, [c_vp, c_u64, c_vp, c_sz, c_vp]),
    "kvs_debug_import_records": (ctypes.c_int, [c_vp, c_u64, c_vp, c_sz, c_vp]),
    "kvs_seq_info": (ctypes.c_int, [c_vp, c_u64, ctypes.POINTER(c_u32), ctypes.POINTER(c_u32),
                                    ctypes.POINTER(c_u32), ctypes.POINTER(c_i32), c_u32]),
    "kvs_set_decode_events": (ctypes.c_int, [c_vp, c_vp, c_vp]),
    "kvs_decode_noalloc": (ctypes.c_int, [c_u32, c_u32, c_u32, c_u32, c_vp, c_u32, c_vp, c_u32,
                                          c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_char_p, c_sz]),
    "kvs_step_count": (c_u64, [c_vp]),
    "kvs_kernel_launches": (c_u64, [c_vp]),
    "kvs_debug_inject": (ctypes.c_int, [c_u32, c_u32]),
    "kvs_debug_chunk_plan": (ctypes.c_int, [ctypes.POINTER(c_u32), c_u32, c_u32, c_u32, c_u32, c_u64, c_u64,
                                            ctypes.POINTER(c_u32), ctypes.POINTER(c_u32),
                                            ctypes.POINTER(c_u32)]),
    "kvs_free_pages": (c_u32, [c_vp]),
    "kvs_check_device": (ctypes.c_int, [c_vp, c_vp]),
}

_lib = None


def lib():
    """The loaded libkvs.so (built by ``paged_kv_cache_flash_gb300.build``)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(
                f"libkvs.so not built ({LIB_PATH}); run `python -m paged_kv_cache_flash_gb300.build`")
        L = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols() -> list:
    return list(_SIGS)


class KvsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        self.code = code
        name = STATUS_NAMES[code] if 0 <= code < len(STATUS_NAMES) else str(code)
        super().__init__(f"KVS_{name}: {msg}")


def _check(ctx, rc):
    if rc != KVS_OK:
        msg = lib().kvs_last_error(ctx).decode(errors="replace")
        raise KvsError(rc, msg)
    return rc


# ----------------------------------------------------------------- config


def make_config(L, Hq, Hkv, d, pool_blocks, max_seqs, max_blocks_per_seq, *, alpha=0.15,
                recency_window=64, weights=(0.25, 0.55, 0.20), cuts=(0.3, 0.6), pool_seed=0,
                staging_pages=16, max_call_blocks=0, kv_dtype=KVS_KV_BF16, k_scale=1.0,
                v_scale=1.0, kivi_groups=0) -> kvs_config:
    return kvs_config(num_layers=L, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                      block_tokens=BLOCK_TOKENS, pool_blocks=pool_blocks, max_seqs=max_seqs,
                      max_blocks_per_seq=max_blocks_per_seq, max_call_blocks=max_call_blocks,
                      staging_pages=staging_pages, alpha=alpha, recency_window=recency_window,
                      kv_dtype=kv_dtype, w_recency=weights[0], w_ema=weights[1],
                      w_anchor=weights[2], cut_lo=cuts[0], cut_hi=cuts[1], pool_seed=pool_seed,
                      k_scale=k_scale, v_scale=v_scale, kivi_groups=kivi_groups)


KVS_FAULT_HOSTALLOC, KVS_FAULT_WAIT = 1, 2


def debug_inject(faults: int = 0, wait_limit_ms: int = 0) -> None:
    """Test hook (process-wide): injected host-side failures; (0, 0) clears."""
    _check(None, lib().kvs_debug_inject(faults, wait_limit_ms))


def debug_chunk_plan(nres, num_layers: int, num_kv_heads: int, workers: int, parts_cap: int,
                     extra_parts: int = 0):
    """Test hook: the decode work-item plan (big, small, tail) of a call whose
    sequences have nres[i] blocks per stream (see kvs_debug_chunk_plan)."""
    arr = (c_u32 * len(nres))(*nres)
    big, small, tail = c_u32(), c_u32(), c_u32()
    _check(None, lib().kvs_debug_chunk_plan(arr, len(nres), num_layers, num_kv_heads, workers, parts_cap,
                                            extra_parts, ctypes.byref(big), ctypes.byref(small),
                                            ctypes.byref(tail)))
    return big.value, small.value, tail.value


def kvs_required_sizes(cfg: kvs_config) -> kvs_sizes:
    sz = kvs_sizes()
    _check(None, lib().kvs_required_sizes(ctypes.byref(cfg), ctypes.byref(sz)))
    return sz


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Context:
    """One pool on the current CUDA device, with torch-allocated buffers."""

    def __init__(self, cfg: kvs_config, device=None):
        import torch
        self.torch = torch
        self.cfg = cfg
        self.device = torch.device(device or "cuda")
        self.sizes = kvs_required_sizes(cfg)
        sz = self.sizes

        def alloc(n):
            return torch.empty(max(int(n), 256), dtype=torch.uint8, device=self.device)
        self.pool = alloc(sz.pool_bytes)
        self.table = alloc(sz.table_bytes)
        self.records = alloc(sz.records_bytes)
        self.mass_buf = alloc(sz.mass_bytes)
        self.workspace = alloc(sz.workspace_bytes)
        self.staging = alloc(sz.staging_bytes)
        self.group_pool = alloc(sz.group_pool_bytes) if sz.group_pool_bytes else None
        bufs = kvs_buffers(self.pool.data_ptr(), self.table.data_ptr(), self.records.data_ptr(),
                           self.mass_buf.data_ptr(), self.workspace.data_ptr(),
                           self.staging.data_ptr(),
                           self.group_pool.data_ptr() if self.group_pool is not None else None)
        h = c_vp()
        with torch.cuda.device(self.device):
            _check(None, lib().kvs_create(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(h)))
        self.h = h
        self.page_bytes = sz.page_bytes
        self._id_arrays = {}        # ctypes id arrays of recurring sequence lists
        self._pinned = {}           # data_ptr -> pinned check of host buffers

    def _ids(self, seq_ids):
        key = tuple(seq_ids)
        arr = self._id_arrays.get(key)
        if arr is None:
            if len(self._id_arrays) > 64:
                self._id_arrays.clear()
            arr = self._id_arrays[key] = (c_u64 * len(key))(*key)
        return arr

    def _host_ok(self, t):
        ok = self._pinned.get(t.data_ptr())
        if ok is None:
            ok = self._pinned[t.data_ptr()] = bool(t.is_pinned())
        return ok

    # -- lifetime --
    def close(self):
        if getattr(self, "h", None):
            lib().kvs_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- calls --
    def seq_add(self, seq_id, parent=-1, shared_prefix_blocks=0, stream=None):
        _check(self.h, lib().kvs_seq_add(self.h, seq_id, parent, shared_prefix_blocks,
                                         _stream_handle(stream)))

    def seq_remove(self, seq_id, stream=None):
        _check(self.h, lib().kvs_seq_remove(self.h, seq_id, _stream_handle(stream)))

    def append_tokens(self, seq_id, k, v, stream=None):
        t = self.torch
        assert k.dtype == t.bfloat16 and v.dtype == t.bfloat16 and k.is_cuda and v.is_cuda
        assert k.is_contiguous() and v.is_contiguous() and k.shape == v.shape
        _check(self.h, lib().kvs_append_tokens(self.h, seq_id, k.shape[0], k.data_ptr(),
                                               v.data_ptr(), _stream_handle(stream)))

    def append_step(self, seq_ids, k, v, stream=None):
        """One token per sequence: k, v CUDA bf16 [nseq][L][Hkv][d]."""
        t = self.torch
        assert k.dtype == t.bfloat16 and v.dtype == t.bfloat16 and k.is_cuda and v.is_cuda
        assert k.is_contiguous() and v.is_contiguous() and k.shape == v.shape
        assert k.shape[0] == len(seq_ids)
        _check(self.h, lib().kvs_append_step(self.h, self._ids(seq_ids), len(seq_ids), k.data_ptr(),
                                             v.data_ptr(), _stream_handle(stream)))

    def decode_step(self, seq_ids, q, out, stream=None):
        t = self.torch
        assert q.dtype == t.bfloat16 and out.dtype == t.float32
        assert q.is_contiguous() and out.is_contiguous() and q.is_cuda and out.is_cuda
        _check(self.h, lib().kvs_decode_step(self.h, self._ids(seq_ids), len(seq_ids), q.data_ptr(),
                                             out.data_ptr(), _stream_handle(stream)))

    def decode_score_step(self, seq_ids, q, out, stream=None):
        """decode_step + score_update, the scoring in the decode epilogue."""
        t = self.torch
        assert q.dtype == t.bfloat16 and out.dtype == t.float32
        assert q.is_contiguous() and out.is_contiguous() and q.is_cuda and out.is_cuda
        _check(self.h, lib().kvs_decode_score_step(self.h, self._ids(seq_ids), len(seq_ids), q.data_ptr(),
                                                   out.data_ptr(), _stream_handle(stream)))

    def score_update(self, stream=None):
        _check(self.h, lib().kvs_score_update(self.h, _stream_handle(stream)))

    def set_alpha(self, alpha):
        _check(self.h, lib().kvs_set_alpha(self.h, alpha))

    def select_and_gather(self, mode, host_dst=None, *, frac=0.0, flags=0, ids=None, slots=None,
                          stream=None, side_stream=None):
        """host_dst: pinned uint8 CPU tensor (or None).  ids: CUDA uint8/int64
        tensor viewed as 16-byte keys; slots: CUDA int32 tensor.  Returns
        (status, kvs_gather_result); KVS_ETRUNC is returned, not raised."""
        a = kvs_gather_args()
        a.mode = mode
        a.flags = flags
        a.frac = frac
        if host_dst is not None:
            assert self._host_ok(host_dst)
            a.host_dst = host_dst.data_ptr()
            a.host_dst_bytes = host_dst.numel() * host_dst.element_size()
        cap = None
        if ids is not None:
            a.ids_dev = ids.data_ptr()
            cap = ids.numel() * ids.element_size() // 16
        if slots is not None:
            a.slot_dev = slots.data_ptr()
            cap = min(cap, slots.numel()) if cap is not None else slots.numel()
        a.ids_capacity = cap or 0
        a.stream = _stream_handle(stream)
        a.side_stream = _stream_handle(side_stream) if side_stream is not None else a.stream
        r = kvs_gather_result()
        rc = lib().kvs_select_and_gather(self.h, ctypes.byref(a), ctypes.byref(r))
        if rc not in (KVS_OK, KVS_ETRUNC):
            _check(self.h, rc)
        return rc, r

    def gather_counts(self):
        """Counts of the latest KVS_GATHER_ASYNC select (waits for them)."""
        r = kvs_gather_result()
        _check(self.h, lib().kvs_gather_counts(self.h, ctypes.byref(r)))
        return r

    def readmit(self, keys, host_src, stream=None):
        n = len(keys)
        arr = (kvs_key * max(n, 1))()
        for i, (s, b) in enumerate(keys):
            arr[i].seq_id = s
            arr[i].block_idx = b
        assert host_src.is_pinned()
        _check(self.h, lib().kvs_readmit(self.h, arr, n, host_src.data_ptr(),
                                         host_src.numel() * host_src.element_size(),
                                         _stream_handle(stream)))

    @staticmethod
    def _plan_out(budget):
        cap = max(budget, 1)
        return (kvs_key * cap)(), (c_dbl * cap)(), (ctypes.c_uint8 * cap)(), c_u32(0)

    @staticmethod
    def _plan_list(keys, blend, cls, n):
        return [(keys[i].seq_id, keys[i].block_idx, int(cls[i]), blend[i]) for i in range(n.value)]

    def prefetch_plan(self, budget, stream=None):
        """[(seq_id, block_idx, class, blend)] of the demoted blocks in fetch
        order, at most `budget`."""
        keys, blend, cls, n = self._plan_out(budget)
        _check(self.h, lib().kvs_prefetch_plan(self.h, budget, keys, blend, cls, ctypes.byref(n),
                                               _stream_handle(stream)))
        return self._plan_list(keys, blend, cls, n)

    def prefetch(self, budget, host_src, stream=None):
        """The plan of prefetch_plan, re-admitted with copies in plan order."""
        assert host_src.is_pinned()
        keys, blend, cls, n = self._plan_out(budget)
        _check(self.h, lib().kvs_prefetch(self.h, budget, host_src.data_ptr(),
                                          host_src.numel() * host_src.element_size(), keys, blend, cls,
                                          ctypes.byref(n), _stream_handle(stream)))
        return self._plan_list(keys, blend, cls, n)

    def debug_set_mass(self, seq_ids, mass, stream=None):
        t = self.torch
        assert mass.dtype == t.float32 and mass.is_cuda and mass.is_contiguous()
        assert mass.shape == (len(seq_ids), self.cfg.max_blocks_per_seq)
        ids = (c_u64 * len(seq_ids))(*seq_ids)
        _check(self.h, lib().kvs_debug_set_mass(self.h, ids, len(seq_ids), mass.data_ptr(),
                                                _stream_handle(stream)))

    def debug_advance(self, steps):
        _check(self.h, lib().kvs_debug_advance(self.h, steps))

    def export_records(self, seq_id, stream=None) -> np.ndarray:
        _, ntok, nb, _ = self.seq_info(seq_id)
        out = np.zeros(max(nb, 1), RECORD_DTYPE)
        _check(self.h, lib().kvs_export_records(self.h, seq_id, out.ctypes.data, nb * 64,
                                                _stream_handle(stream)))
        return out[:nb]

    def debug_import_records(self, seq_id, recs: np.ndarray, stream=None):
        """Test hook: overwrites the sequence's records (RECORD_DTYPE, block order)."""
        recs = np.ascontiguousarray(recs)
        assert recs.dtype.itemsize == 64
        _check(self.h, lib().kvs_debug_import_records(self.h, seq_id, recs.ctypes.data, recs.nbytes,
                                                      _stream_handle(stream)))

    def seq_info(self, seq_id):
        """(slot, n_tokens, n_blocks, table)"""
        sl, nt, nb = c_u32(), c_u32(), c_u32()
        _check(self.h, lib().kvs_seq_info(self.h, seq_id, ctypes.byref(sl), ctypes.byref(nt),
                                          ctypes.byref(nb), None, 0))
        table = (c_i32 * max(nb.value, 1))()
        _check(self.h, lib().kvs_seq_info(self.h, seq_id, None, None, None, table, nb.value))
        return sl.value, nt.value, nb.value, list(table)[:nb.value]

    def set_decode_events(self, start=None, stop=None):
        """torch.cuda.Event pair recorded around the decode kernel (None: off)."""
        a = start.cuda_event if start is not None else None
        b = stop.cuda_event if stop is not None else None
        _check(self.h, lib().kvs_set_decode_events(self.h, a, b))

    def step_count(self) -> int:
        return lib().kvs_step_count(self.h)

    def kernel_launches(self) -> int:
        return lib().kvs_kernel_launches(self.h)

    def free_pages(self) -> int:
        return lib().kvs_free_pages(self.h)

    def check_device(self, stream=None):
        _check(self.h, lib().kvs_check_device(self.h, _stream_handle(stream)))

    def mass(self):
        """Mass buffer as a float32 [max_seqs][max_blocks_per_seq] tensor view
        (row = sequence slot, see seq_info)."""
        return self.mass_buf[: self.sizes.mass_bytes].view(self.torch.float32).view(
            self.cfg.max_seqs, self.cfg.max_blocks_per_seq)

    def group_bytes_of(self, group_page: int):
        """Bytes of a 2-bit group page (a CUDA uint8 view)."""
        gb = self.sizes.group_page_bytes
        return self.group_pool[group_page * gb:(group_page + 1) * gb]

    def page_bytes_of(self, page: int):
        """Bytes of a physical page (a CUDA uint8 view)."""
        pb = self.page_bytes
        return self.pool[page * pb:(page + 1) * pb]
