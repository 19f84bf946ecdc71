"""Python binding of libkvs, the sm_103a sparse KV-cache decode step library.

Argument marshalling only: every function forwards to the C ABI in include/kvs.h (same names,
same meaning), passing device pointers from torch tensors and the current CUDA stream.  There is
no fallback: when libkvs.so is missing or a call fails, an exception is raised.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvs.so")

STATUS = {0: "KVS_OK", 1: "KVS_ERR_INVALID_ARG", 2: "KVS_ERR_CUDA", 3: "KVS_ERR_CAPACITY", 4: "KVS_ERR_TIMEOUT",
          5: "KVS_ERR_HOST_MEM", 6: "KVS_ERR_NOT_SUPPORTED", 7: "KVS_ERR_BAD_INDEX"}


class KvsError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class KvsConfig(ctypes.Structure):
    _fields_ = [("n_req", ctypes.c_int), ("n_layer", ctypes.c_int), ("n_q_head", ctypes.c_int),
                ("n_kv_head", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
                ("v_shares_k", ctypes.c_int), ("block_size", ctypes.c_int), ("max_ctx", ctypes.c_int),
                ("budget_blocks", ctypes.c_int), ("n_sink", ctypes.c_int), ("n_recent", ctypes.c_int),
                ("cap_blocks", ctypes.c_int), ("max_score_q", ctypes.c_int), ("lookahead", ctypes.c_int),
                ("max_prefetch", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("wait_timeout_us", ctypes.c_uint), ("evict_policy", ctypes.c_int), ("score_mode", ctypes.c_int),
                ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]

EVICT_POLICY = {"lru": 0, "importance": 1}
SCORE_MODE = {"mean": 0, "bound": 1}
KV_DTYPE = {"bf16": 0, "fp8": 1}


class KvsStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_ulonglong) for n in
                ("hits", "misses", "evictions", "prefetched", "prefetch_hits", "pin_fallbacks", "bytes_fetched")]


STATS_FIELDS = [f[0] for f in KvsStats._fields_]

_lib = None

# name -> (restype, argtypes)
_P, _I, _U = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
_SIGS = {
    "kvs_version": (ctypes.c_char_p, []),
    "kvs_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(KvsConfig)]),
    "kvs_create": (_I, [ctypes.POINTER(KvsConfig), _P, ctypes.c_size_t, ctypes.POINTER(_P)]),
    "kvs_destroy": (_I, [_P]),
    "kvs_bind_host_kv": (_I, [_P, _P, _P]),
    "kvs_index_build": (_I, [_P, _I, _P, _P, _P]),
    "kvs_score_blocks": (_I, [_P, _I, _P, _I, _P, _P, _P, _P]),
    "kvs_topk_select": (_I, [_P, _P, _P, _P, _P, _P]),
    "kvs_cache_update": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P]),
    "kvs_snapshot_bytes": (ctypes.c_size_t, [ctypes.POINTER(KvsConfig)]),
    "kvs_cache_snapshot": (_I, [_P, _I, _P, _P]),
    "kvs_cache_restore": (_I, [_P, _I, _P, _P, _P]),
    "kvs_sparse_decode_attn": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P]),
    "kvs_decode_step": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "kvs_join": (_I, [_P, _P]),
    "kvs_layer_prefetch": (_I, [_P, _I, _P, _P, _P, _P, _P]),
    "kvs_advance_ctx": (_I, [_P, _P, _P]),
    "kvs_append": (_I, [_P, _I, _P, _P, _P, _P, _P]),
    "kvs_cache_export": (_I, [_P, _I, _P, _P, _P, _P]),
    "kvs_slot_pools": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "kvs_poll_error": (_I, [_P, ctypes.POINTER(_I)]),
    "kvs_kernel_timer_arm": (_I, [_P, _I, _I]),
    "kvs_kernel_timer_read": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I)]),
    "kvs_launch_count": (ctypes.c_ulonglong, [_P]),
    "kvs_select_blocks_noalloc": (_I, [ctypes.POINTER(KvsConfig), _P, _I, _P, _P, _P, _P, _P, _P]),
    "kvs_probe_host_read": (_I, [_P, ctypes.c_size_t, _P, _I, _I, _I, _I, _P, _P]),
    "kvs_quantize_e4m3": (_I, [_P, _P, ctypes.c_size_t, ctypes.c_float, _P]),
}

KERNEL_IDS = {"score": 1, "topk": 2, "update": 3, "fetch": 4, "attn": 5, "prefetch": 6, "append": 7, "index": 8}


def lib():
    """Load libkvs.so (built by __graft_entry__.build() / sparse_kv_cache_decode_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvs.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise KvsError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if not isinstance(stream, int) else stream


def make_config(w, max_score_q: int | None = None, max_prefetch: int = 0, wait_timeout_us: int = 0) -> KvsConfig:
    """kvs_config of a workload description (anything with the workload.Workload fields)."""
    return KvsConfig(w.n_req, w.n_layer, w.n_q_head, w.n_kv_head, w.d_k, w.d_v, int(w.v_shares_k), w.block_size,
                     w.max_ctx, w.budget_blocks, w.n_sink, w.n_recent, w.cap_blocks,
                     max_score_q if max_score_q is not None else max(1, w.n_score_q), int(w.lookahead), max_prefetch,
                     float(w.softmax_scale), wait_timeout_us, EVICT_POLICY[getattr(w, "evict_policy", "lru")],
                     SCORE_MODE[getattr(w, "score_mode", "mean")], KV_DTYPE[getattr(w, "kv_dtype", "bf16")],
                     float(getattr(w, "k_scale", 1.0)), float(getattr(w, "v_scale", 1.0)))


class Context:
    """A kvs_ctx with its device workspace (allocated through torch) and its bound host history."""

    def __init__(self, cfg: KvsConfig, device: int = 0):
        import torch
        self.cfg = cfg
        self.L = lib()
        nbytes = self.L.kvs_workspace_bytes(ctypes.byref(cfg))
        if nbytes == 0:
            raise KvsError(1, "kvs_workspace_bytes")
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=f"cuda:{device}")
        base = self.workspace.data_ptr()
        aligned = (base + 255) // 256 * 256
        h = _P()
        _check(self.L.kvs_create(ctypes.byref(cfg), aligned, nbytes, ctypes.byref(h)), "kvs_create")
        self.h = h
        self.nb_max = (cfg.max_ctx + cfg.block_size - 1) // cfg.block_size
        self.units = cfg.n_req * cfg.n_kv_head
        self._host = None

    def close(self):
        if getattr(self, "h", None):
            self.L.kvs_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ C-ABI forwards
    def bind_host_kv(self, h_k, h_v=None):
        self._host = (h_k, h_v)
        _check(self.L.kvs_bind_host_kv(self.h, _ptr(h_k), _ptr(h_v)), "kvs_bind_host_kv")

    def index_build(self, layer, index, ctx_len, stream=None):
        _check(self.L.kvs_index_build(self.h, layer, _ptr(index), _ptr(ctx_len), _stream(stream)), "kvs_index_build")

    def score_blocks(self, layer, score_q, nq, index, ctx_len, scores, stream=None):
        _check(self.L.kvs_score_blocks(self.h, layer, _ptr(score_q), nq, _ptr(index), _ptr(ctx_len), _ptr(scores),
                                       _stream(stream)), "kvs_score_blocks")

    def topk_select(self, scores, ctx_len, sel, nsel, stream=None):
        _check(self.L.kvs_topk_select(self.h, _ptr(scores), _ptr(ctx_len), _ptr(sel), _ptr(nsel), _stream(stream)),
               "kvs_topk_select")

    def cache_update(self, layer, sel, nsel, ctx_len, slot_of_sel, stats=None, stream=None, scores=None):
        _check(self.L.kvs_cache_update(self.h, layer, _ptr(sel), _ptr(nsel), _ptr(ctx_len), _ptr(slot_of_sel),
                                       _ptr(scores), _ptr(stats), _stream(stream)), "kvs_cache_update")

    def snapshot_bytes(self) -> int:
        return int(self.L.kvs_snapshot_bytes(ctypes.byref(self.cfg)))

    def cache_snapshot(self, layer, snap, stream=None):
        _check(self.L.kvs_cache_snapshot(self.h, layer, _ptr(snap), _stream(stream)), "kvs_cache_snapshot")

    def cache_restore(self, layer, snap, ctx_len, stream=None):
        _check(self.L.kvs_cache_restore(self.h, layer, _ptr(snap), _ptr(ctx_len), _stream(stream)),
               "kvs_cache_restore")

    def sparse_decode_attn(self, layer, q, sel, slot_of_sel, nsel, ctx_len, out, stream=None):
        _check(self.L.kvs_sparse_decode_attn(self.h, layer, _ptr(q), _ptr(sel), _ptr(slot_of_sel), _ptr(nsel),
                                             _ptr(ctx_len), _ptr(out), _stream(stream)), "kvs_sparse_decode_attn")

    def decode_step(self, layer, q, score_q, nq, index, ctx_len, out, stats=None, k_new=None, v_new=None,
                    sel_out=None, nsel_out=None, stream=None, copy_stream=None):
        cs = None if copy_stream is None else _stream(copy_stream)
        _check(self.L.kvs_decode_step(self.h, layer, _ptr(q), _ptr(score_q), nq, _ptr(k_new), _ptr(v_new),
                                      _ptr(index), _ptr(ctx_len), _ptr(out), _ptr(stats), _ptr(sel_out),
                                      _ptr(nsel_out), _stream(stream), cs), "kvs_decode_step")

    def join(self, stream=None):
        _check(self.L.kvs_join(self.h, _stream(stream)), "kvs_join")

    def layer_prefetch(self, dst_layer, hint_sel, hint_nsel, ctx_len, stats=None, stream=None):
        _check(self.L.kvs_layer_prefetch(self.h, dst_layer, _ptr(hint_sel), _ptr(hint_nsel), _ptr(ctx_len),
                                         _ptr(stats), _stream(stream)), "kvs_layer_prefetch")

    def advance_ctx(self, ctx_len, stream=None):
        _check(self.L.kvs_advance_ctx(self.h, _ptr(ctx_len), _stream(stream)), "kvs_advance_ctx")

    def append(self, layer, k_new, v_new, index, ctx_len, stream=None):
        _check(self.L.kvs_append(self.h, layer, _ptr(k_new), _ptr(v_new), _ptr(index), _ptr(ctx_len),
                                 _stream(stream)), "kvs_append")

    def cache_export(self, layer):
        import numpy as np
        c = self.cfg
        b2s = np.empty((self.units, self.nb_max), np.int32)
        s2b = np.empty((self.units, c.cap_blocks), np.int32)
        st = np.empty((self.units, c.cap_blocks), np.uint32)
        clk = np.empty(self.units, np.uint32)
        _check(self.L.kvs_cache_export(self.h, layer, b2s.ctypes.data, s2b.ctypes.data, st.ctypes.data,
                                       clk.ctypes.data), "kvs_cache_export")
        return b2s, s2b, st, clk

    def slot_pools(self, layer):
        k, v = _P(), _P()
        _check(self.L.kvs_slot_pools(self.h, layer, ctypes.byref(k), ctypes.byref(v)), "kvs_slot_pools")
        return k.value, v.value

    def slot_pool_tensors(self, layer):
        """Views (int16 bf16 patterns, or uint8 E4M3 codes) of one layer's slot pools inside the workspace tensor:
        K [units][C][bs][d_k] and V [units][C][bs][d_v] (None when V shares the K row)."""
        c = self.cfg
        kp, vp = self.slot_pools(layer)
        base = self.workspace.data_ptr()

        torch = __import__("torch")
        fp8 = c.kv_dtype == KV_DTYPE["fp8"]

        def view(ptr, d):
            n = self.units * c.cap_blocks * c.block_size * d * (1 if fp8 else 2)
            off = ptr - base
            return self.workspace[off: off + n].view(dtype=torch.uint8 if fp8 else torch.int16).view(
                self.units, c.cap_blocks, c.block_size, d)

        return view(kp, c.d_k), (None if vp is None else view(vp, c.d_v))

    def kernel_timer_arm(self, kernel: str, capacity: int):
        _check(self.L.kvs_kernel_timer_arm(self.h, KERNEL_IDS[kernel], capacity), "kvs_kernel_timer_arm")

    def kernel_timer_read(self, kernel: str):
        ms, n = ctypes.c_double(), _I()
        _check(self.L.kvs_kernel_timer_read(self.h, KERNEL_IDS[kernel], ctypes.byref(ms), ctypes.byref(n)),
               "kvs_kernel_timer_read")
        return ms.value, n.value

    def launch_count(self) -> int:
        return int(self.L.kvs_launch_count(self.h))

    def poll_error(self) -> int:
        st = _I()
        _check(self.L.kvs_poll_error(self.h, ctypes.byref(st)), "kvs_poll_error")
        return st.value


_MBIND_NR = {"aarch64": 235, "x86_64": 237}


def bind_local_node(addr: int, length: int):
    """Give [addr, addr + length) an explicit memory policy of this process: preferred node = the
    NUMA node of the CPU the caller runs on (mbind, MPOL_PREFERRED).  A range with an explicit
    policy is left alone by automatic NUMA balancing, which otherwise samples it with hinting
    faults.  Only this process's mapping changes.  Returns the node, or None when the call is not
    available."""
    import os
    import platform
    nr = _MBIND_NR.get(platform.machine())
    if nr is None:
        return None
    try:
        cpu = min(os.sched_getaffinity(0))
        nodes = [d for d in os.listdir(f"/sys/devices/system/cpu/cpu{cpu}") if d.startswith("node") and d[4:].isdigit()]
        node = int(nodes[0][4:]) if nodes else 0
    except OSError:
        return None
    mask = (ctypes.c_ulong * 16)()
    mask[node // 64] = 1 << (node % 64)
    libc = ctypes.CDLL(None, use_errno=True)
    libc.syscall.restype = ctypes.c_long
    rc = libc.syscall(ctypes.c_long(nr), ctypes.c_void_p(addr), ctypes.c_ulong(length), ctypes.c_int(1),  # MPOL_PREFERRED
                      mask, ctypes.c_ulong(16 * 64), ctypes.c_uint(0))
    return node if rc == 0 else None


def numa_vmstat() -> dict:
    """Counters of /proc/vmstat about huge-page splits and NUMA balancing (diagnostics)."""
    keys = ("thp_split_pmd", "thp_split_page", "numa_hint_faults", "numa_pages_migrated", "numa_pte_updates",
            "thp_migration_success", "thp_migration_fail", "thp_migration_split", "pgmigrate_fail")
    out = {}
    try:
        with open("/proc/vmstat") as f:
            for ln in f:
                k, v = ln.split()
                if k in keys:
                    out[k] = int(v)
    except OSError:
        pass
    return out


class HostArray:
    """Page-locked, device-mapped host memory for the KV history, backed by transparent huge
    pages: an anonymous mmap aligned to 512 MiB and advised MADV_HUGEPAGE, then registered with
    cudaHostRegister (portable | mapped).  Large pages keep the GPU's translations of scattered
    block fetches cheap.  Fill it (first touch) before calling register()."""

    HUGE_ALIGN = 1 << 29

    def __init__(self, shape, dtype=None, huge: bool = True, local_node: bool = False):
        import mmap
        import torch
        dtype = dtype or torch.int16
        self.nbytes = int(math.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        align = self.HUGE_ALIGN if huge else mmap.PAGESIZE
        self._mm = mmap.mmap(-1, self.nbytes + align, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        base = ctypes.addressof(ctypes.c_char.from_buffer(self._mm))
        off = (-base) % align
        length = (self.nbytes + mmap.PAGESIZE - 1) // mmap.PAGESIZE * mmap.PAGESIZE
        if huge and hasattr(mmap, "MADV_HUGEPAGE"):
            self._mm.madvise(mmap.MADV_HUGEPAGE, off, length)
        self.node = bind_local_node(base + off, length) if local_node else None
        self.tensor = torch.frombuffer(self._mm, dtype=torch.uint8, count=self.nbytes, offset=off).view(dtype).view(
            *shape)
        self._registered = False

    def huge_fraction(self) -> float:
        """Fraction of this array backed by transparent huge pages (from /proc/self/smaps)."""
        lo = self.tensor.data_ptr()
        hi = lo + self.nbytes
        huge = 0
        try:
            with open("/proc/self/smaps") as f:
                cur = None
                for ln in f:
                    head = ln.split()[0]
                    if "-" in head and ":" not in head:
                        a, b = (int(x, 16) for x in head.split("-"))
                        cur = (a, b) if (a < hi and b > lo) else None
                    elif cur is not None and ln.startswith("AnonHugePages:"):
                        huge += int(ln.split()[1]) * 1024
        except OSError:
            return 0.0
        return min(1.0, huge / self.nbytes)

    def register(self):
        import torch
        rc = torch.cuda.cudart().cudaHostRegister(self.tensor.data_ptr(), self.nbytes, 3)
        if int(rc) != 0:
            raise RuntimeError(f"cudaHostRegister failed ({rc})")
        self._registered = True
        return self

    MADV_COLLAPSE = 25   # Linux >= 6.1: map the range with huge pages again, synchronously

    def recollapse(self) -> float:
        """Map the array with huge pages again after some of its huge-page mappings were split
        (the pages stay in place and keep their contents): unregister, advise MADV_COLLAPSE,
        register again.  Returns the huge fraction afterwards; callers bind the history anew."""
        import mmap
        import torch
        was = self._registered
        if was:
            torch.cuda.cudart().cudaHostUnregister(self.tensor.data_ptr())
            self._registered = False
        base = ctypes.addressof(ctypes.c_char.from_buffer(self._mm))
        off = self.tensor.data_ptr() - base
        try:
            self._mm.madvise(self.MADV_COLLAPSE, off, (self.nbytes + mmap.PAGESIZE - 1) // mmap.PAGESIZE * mmap.PAGESIZE)
        except OSError:
            pass
        if was:
            self.register()
        return self.huge_fraction()

    def close(self):
        import torch
        if self._registered:
            torch.cuda.cudart().cudaHostUnregister(self.tensor.data_ptr())
            self._registered = False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pinned_host_history(shape, fill, min_huge: float = 0.95, local_node: bool = False):
    """Host history of the given shape, filled by fill(tensor) and page-locked for the device.

    Prefers a HostArray on transparent huge pages (fewest GPU translation misses on scattered
    block fetches); when the kernel could not back it with huge pages, falls back to
    cudaHostAlloc memory (torch pin_memory).  Returns (tensor, keepalive, description)."""
    import torch
    arr = HostArray(shape, local_node=local_node)
    fill(arr.tensor)
    frac = arr.huge_fraction()
    if frac >= min_huge:
        arr.register()
        return arr.tensor, arr, f"mmap + transparent huge pages ({frac:.0%}) + cudaHostRegister"
    t = torch.empty(shape, dtype=arr.tensor.dtype, pin_memory=True)
    t.copy_(arr.tensor)
    del arr
    return t, None, f"cudaHostAlloc (huge pages covered only {frac:.0%})"


def select_blocks_noalloc(cfg: KvsConfig, score_q, nq: int, index_layer, ctx_len, sel, nsel, status=None,
                          stream=None) -> None:
    """kvs_select_blocks_noalloc: one layer's block selection with no device allocation (the
    block scores live in a fixed device array inside the library)."""
    _check(lib().kvs_select_blocks_noalloc(ctypes.byref(cfg), _ptr(score_q), nq, _ptr(index_layer), _ptr(ctx_len),
                                           _ptr(sel), _ptr(nsel), _ptr(status), _stream(stream)),
           "kvs_select_blocks_noalloc")


def probe_host_read(h_base, region_bytes: int, offsets, item_bytes: int, n_ctas: int, threads: int, sink,
                    stream=None) -> None:
    """kvs_probe_host_read: SM zero-copy reads of items at device-resident byte offsets (int64)
    from page-locked, device-mapped host memory (diagnostics for the host-link peak)."""
    _check(lib().kvs_probe_host_read(_ptr(h_base), region_bytes, _ptr(offsets), int(offsets.numel()), item_bytes,
                                     n_ctas, threads, _ptr(sink), _stream(stream)), "kvs_probe_host_read")


def quantize_e4m3(src, dst, scale: float, stream=None) -> None:
    """kvs_quantize_e4m3 on device tensors: dst (uint8, n) = E4M3 codes of src (bf16 patterns, n) / scale."""
    n = src.numel()
    if dst.numel() != n:
        raise ValueError("quantize_e4m3: sizes differ")
    _check(lib().kvs_quantize_e4m3(_ptr(src), _ptr(dst), n, float(scale), _stream(stream)), "kvs_quantize_e4m3")


def quantize_history_e4m3(src_host, dst_host, scale: float, chunk: int = 1 << 28) -> None:
    """E4M3 codes of a host bf16 history into a host uint8 array of the same shape, through the GPU
    in chunks (each chunk copied in, quantised by kvs_quantize_e4m3, copied back)."""
    import torch
    s = src_host.view(-1)
    d = dst_host.view(-1)
    if s.numel() != d.numel():
        raise ValueError("quantize_history_e4m3: sizes differ")
    n = s.numel()
    step = min(chunk, n)
    bs = torch.empty(step, dtype=torch.int16, device="cuda")
    bd = torch.empty(step, dtype=torch.uint8, device="cuda")
    for i in range(0, n, step):
        m = min(step, n - i)
        bs[:m].copy_(s[i:i + m])
        quantize_e4m3(bs[:m], bd[:m], scale)
        d[i:i + m].copy_(bd[:m])
    torch.cuda.synchronize()


def version() -> str:
    return lib().kvs_version().decode()
