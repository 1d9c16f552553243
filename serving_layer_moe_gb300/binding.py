"""ctypes binding of libmoecache.so (argument marshalling only).

Every step of the MoE layer runs in the library's CUDA kernels; this module
only turns torch tensors into device pointers and C structs.  It never falls
back to anything: if the library is missing it raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoecache.so")

MOE_F32, MOE_BF16, MOE_FP8E4M3_B128, MOE_NVFP4, MOE_MXFP4 = 0, 1, 2, 3, 4
DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16, "fp8": MOE_FP8E4M3_B128, "nvfp4": MOE_NVFP4, "mxfp4": MOE_MXFP4}
STATUS = {0: "MOE_OK", 1: "MOE_EINVAL", 2: "MOE_ENOMEM", 3: "MOE_ECUDA", 4: "MOE_ECAPACITY",
          5: "MOE_EBUSY", 6: "MOE_EDEVICE"}

# exported symbols of include/moe_cache.h
SYMBOLS = ("moe_cache_create", "moe_cache_destroy", "moe_cache_resize", "moe_layer_decode",
           "moe_layer_prefill", "moe_cache_get_state", "moe_cache_get_plan", "moe_cache_info",
           "moe_cache_profile", "moe_cache_set_prefill_prefetch", "moe_cache_set_cpu_branch", "bench_bw",
           "moe_layer_ffn_noalloc", "moe_last_error")

# moe_cpu_branch_fn: (user, layer, T, x_host, topk_ids_host, slot_map_host, cpu_part_host)
CPU_BRANCH_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                 ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_float))


class MoEConfigC(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("top_k", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("max_fetch", ctypes.c_int32), ("wdtype", ctypes.c_int32), ("adtype", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("bw_pcie_mbps", ctypes.c_uint32),
                ("bw_cpu_mbps", ctypes.c_uint32), ("device", ctypes.c_int32),
                ("max_prefill_tokens", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load_library():
    """Load the in-tree libmoecache.so and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; build it with serving_layer_moe_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, U32, U64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64
    lib.moe_cache_create.argtypes = [ctypes.POINTER(MoEConfigC), P, U64, P, P, U64, ctypes.POINTER(P)]
    lib.moe_cache_destroy.argtypes = [P]
    lib.moe_cache_resize.argtypes = [P, U64]
    lib.moe_layer_decode.argtypes = [P, I32, I32, P, P, P, P, P, P, P]
    lib.moe_layer_prefill.argtypes = [P, I32, I32, P, P, P, P, P]
    lib.moe_cache_get_state.argtypes = [P, P, P, P, P, P]
    lib.moe_cache_get_plan.argtypes = [P, P, P, P, P]
    lib.moe_cache_info.argtypes = [P, P]
    lib.moe_cache_profile.argtypes = [P, I32, P, P]
    lib.moe_cache_set_prefill_prefetch.argtypes = [P, I32]
    lib.moe_cache_set_cpu_branch.argtypes = [P, CPU_BRANCH_FN, P]
    lib.bench_bw.argtypes = [I32, U64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                             ctypes.POINTER(I32)]
    lib.moe_layer_ffn_noalloc.argtypes = [I32, I32, I32, I32, I32, I32, P, I32, P, P, P, P, P]
    lib.moe_last_error.restype = ctypes.c_char_p
    for name in SYMBOLS[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise MoEError(status, load_library().moe_last_error().decode())


def _ptr(t) -> int | None:
    """Device or host address of a torch tensor / numpy array (None stays NULL)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        if not t.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays passed to the library must be C-contiguous")
        return t.ctypes.data
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


class MoECache:
    """One LRU cache of whole experts on one GPU, a slot per resident (layer, expert) (libmoecache.so).

    host_pool: page-locked or pageable host memory (torch uint8 tensor or numpy
    array) holding the expert blobs; it is kept referenced by this object.
    """

    def __init__(self, *, L, E, H, I, top_k, max_tokens, wdtype, adtype, host_pool, n_slots,
                 blob_offsets=None, shared=None, max_fetch=-1, bw_pcie_mbps=1, bw_cpu_mbps=0,
                 device=0, max_prefill_tokens=0):
        lib = load_library()
        self._pool = host_pool
        self._shared = shared
        cfg = MoEConfigC(L, E, H, I, top_k, max_tokens, max_fetch, DTYPES.get(wdtype, wdtype),
                         DTYPES.get(adtype, adtype), 1 if shared is not None else 0, int(bw_pcie_mbps),
                         int(bw_cpu_mbps), device, max_prefill_tokens)
        offs = None if blob_offsets is None else np.ascontiguousarray(blob_offsets, dtype=np.uint64)
        nbytes = host_pool.nbytes if isinstance(host_pool, np.ndarray) else host_pool.numel() * host_pool.element_size()
        handle = ctypes.c_void_p()
        _check(lib.moe_cache_create(ctypes.byref(cfg), _ptr(host_pool), nbytes, _ptr(offs), _ptr(shared),
                                    int(n_slots), ctypes.byref(handle)))
        self._h = handle
        self.L, self.E, self.H, self.I, self.k = L, E, H, I, top_k
        self._adtype = DTYPES.get(adtype, adtype)
        info = self.info()
        self.S, self.C, self.K = int(info[0]), int(info[1]), int(info[2])

    # -- calls ----------------------------------------------------------------
    def decode(self, layer, x, topk_ids, topk_w, out, cpu_part=None, slot_map=None, stream=None):
        T = topk_ids.shape[0]
        _check(load_library().moe_layer_decode(self._h, layer, T, _ptr(x), _ptr(topk_ids), _ptr(topk_w),
                                               _ptr(cpu_part), _ptr(out), _ptr(slot_map), _stream(stream)))

    def decode_ptrs(self, layer, T, x, ids, w, cpu_part, out, slot_map, stream):
        """decode() on raw addresses (for tight loops)."""
        _check(load_library().moe_layer_decode(self._h, layer, T, x, ids, w, cpu_part, out, slot_map, stream))

    def decode_from_host(self, layer, x_host, ids_host, w_host, out_host, cpu_part=None, stream=None):
        """decode() on page-locked host tensors: the copies in (cpu_part too, if it
        is on the host), the call and the copy of the output back, all enqueued on
        one stream (`stream`, else torch's current stream).  Returns out_host once
        the copy back is enqueued: synchronise that stream before reading it."""
        import torch
        dev = torch.device("cuda", torch.cuda.current_device())
        if stream is None:
            s = torch.cuda.current_stream(dev)
        elif isinstance(stream, torch.cuda.Stream):
            s = stream
        else:
            s = torch.cuda.ExternalStream(int(stream), device=dev)
        with torch.cuda.stream(s):
            x = x_host.to(dev, non_blocking=True)
            ids = ids_host.to(dev, non_blocking=True)
            w = w_host.to(dev, non_blocking=True)
            cp = None if cpu_part is None else cpu_part.to(dev, non_blocking=True)
            out = torch.empty(out_host.shape, dtype=torch.float32, device=dev)
            self.decode(layer, x, ids, w, out, cpu_part=cp, stream=s)
            out_host.copy_(out, non_blocking=True)
        return out_host

    def prefill(self, layer, x, topk_ids, topk_w, out, stream=None):
        T = topk_ids.shape[0]
        _check(load_library().moe_layer_prefill(self._h, layer, T, _ptr(x), _ptr(topk_ids), _ptr(topk_w),
                                                _ptr(out), _stream(stream)))

    def set_prefill_prefetch(self, on: bool):
        """The second prefill buffer (the next layer loads during this one's GEMMs) on or off."""
        _check(load_library().moe_cache_set_prefill_prefetch(self._h, 1 if on else 0))

    def set_cpu_branch(self, fn):
        """Register fn(layer, T, x, topk_ids, slot_map, cpu_part) as the CPU branch of every
        decode call (None removes it).  The library calls it from a CUDA host node with
        numpy views of its page-locked staging: x [T, H] (uint16 bf16 bits or float32),
        topk_ids and slot_map [T, k] int32, and cpu_part [T, k, H] float32, which fn fills
        wherever slot_map < 0.  It runs on a driver thread: wait for a decode call through
        this library (state(), which releases the interpreter lock), not through calls that
        hold the lock while the stream drains."""
        lib = load_library()
        if fn is None:
            _check(lib.moe_cache_set_cpu_branch(self._h, CPU_BRANCH_FN(), None))
            self._cpu_cb = None
            return
        H, k = self.H, self.k
        xdt = np.float32 if self._adtype == MOE_F32 else np.uint16

        def trampoline(_user, layer, T, x_ptr, ids_ptr, sm_ptr, cp_ptr):
            x = np.ctypeslib.as_array(ctypes.cast(x_ptr, ctypes.POINTER(
                ctypes.c_float if xdt is np.float32 else ctypes.c_uint16)), shape=(T, H))
            ids = np.ctypeslib.as_array(ids_ptr, shape=(T, k))
            sm = np.ctypeslib.as_array(sm_ptr, shape=(T, k))
            cp = np.ctypeslib.as_array(cp_ptr, shape=(T, k, H))
            fn(int(layer), int(T), x, ids, sm, cp)

        cb = CPU_BRANCH_FN(trampoline)
        _check(lib.moe_cache_set_cpu_branch(self._h, cb, None))
        self._cpu_cb = cb   # the library holds the pointer: keep the callback alive

    def resize(self, n_slots):
        _check(load_library().moe_cache_resize(self._h, int(n_slots)))
        self.C = int(self.info()[1])

    # -- readout ------------------------------------------------------------------
    def state(self):
        s2e = np.empty(self.C, np.int32)
        st = np.empty(self.C, np.uint64)
        e2s = np.empty(self.L * self.E, np.int32)
        cnt = np.empty(8, np.uint64)
        clk = np.empty(1, np.uint64)
        _check(load_library().moe_cache_get_state(self._h, _ptr(s2e), _ptr(st), _ptr(e2s), _ptr(cnt), _ptr(clk)))
        return s2e, st, e2s, cnt, int(clk[0])

    def plan(self, T=None):
        sc = np.empty(8, np.int32)
        v = np.empty(max(self.K, 1), np.int32)
        f = np.empty(2 * max(self.K, 1), np.int32)
        y = None if T is None else np.empty((T, self.k, self.H), np.float32)
        _check(load_library().moe_cache_get_plan(self._h, _ptr(sc), _ptr(v), _ptr(f), _ptr(y)))
        out = dict(layer=int(sc[0]), u=int(sc[1]), h=int(sc[2]), m=int(sc[3]), q=int(sc[4]),
                   n_cpu=int(sc[5]), n_gpu=int(sc[6]), victims=v[: self.K].tolist(),
                   fills=[(int(f[2 * i]), int(f[2 * i + 1])) for i in range(int(sc[4]))])
        if y is not None:
            out["y"] = y
        return out

    PROFILE_KINDS = ("control", "fill", "gemv_resident", "down_filled", "down_combine",
                     "prefill_control", "prefill_load", "prefill_gemm")

    def profile_start(self):
        _check(load_library().moe_cache_profile(self._h, 1, None, None))

    def _profile(self, mode):
        ms = np.zeros(8, np.float64)
        n = np.zeros(8, np.uint64)
        _check(load_library().moe_cache_profile(self._h, mode, _ptr(ms), _ptr(n)))
        return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(self.PROFILE_KINDS)}

    def profile_stop(self):
        """{kind: (milliseconds, timed launches)} since profile_start(); stops and resets."""
        return self._profile(0)

    def profile_pause(self):
        """Keep the pairs recorded so far (e.g. captured into a graph); record no new ones."""
        _check(load_library().moe_cache_profile(self._h, 3, None, None))

    def profile_read(self):
        """{kind: (milliseconds, launches)} over the recorded pairs, without resetting."""
        return self._profile(2)

    def info(self):
        info = np.empty(8, np.uint64)
        _check(load_library().moe_cache_info(self._h, _ptr(info)))
        return info

    def close(self):
        if getattr(self, "_h", None):
            load_library().moe_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bench_bw(device: int, expert_bytes: int):
    """(B_P GB/s, B_H GB/s, recommend_hybrid) measured on `device`."""
    lib = load_library()
    bp, bh, rec = ctypes.c_double(), ctypes.c_double(), ctypes.c_int32()
    _check(lib.bench_bw(device, int(expert_bytes), ctypes.byref(bp), ctypes.byref(bh), ctypes.byref(rec)))
    return bp.value, bh.value, bool(rec.value)


def blob_bytes(wdtype, H: int, I: int) -> int:
    """S, the bytes of one expert blob in the bank layout moe_cache.h states."""
    wd = DTYPES.get(wdtype, wdtype)
    HI = H * I
    if wd == MOE_F32:
        return 12 * HI
    if wd == MOE_BF16:
        return 6 * HI
    if wd == MOE_FP8E4M3_B128:
        return 3 * HI + 4 * ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128))
    if wd == MOE_NVFP4:
        return 3 * HI // 2 + 3 * HI // 16 + 16
    if wd == MOE_MXFP4:
        return 3 * HI // 2 + 3 * HI // 32
    raise ValueError(f"unknown weight dtype {wdtype!r}")


def _nbytes(t) -> int:
    return t.nbytes if isinstance(t, np.ndarray) else t.numel() * t.element_size()


def _check_noalloc_args(experts, x, topk_ids, topk_w, out, E, H, I, top_k, wdtype, adtype):
    """Refuse arguments the kernels would read or write out of bounds (ValueError)."""
    import torch
    wd, ad = DTYPES.get(wdtype, wdtype), DTYPES.get(adtype, adtype)
    if ad not in (MOE_F32, MOE_BF16):
        raise ValueError(f"adtype must be f32 or bf16, not {adtype!r}")
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2 or topk_ids.shape[1] != top_k:
        raise ValueError(f"topk_ids must be int32 [T, {top_k}], got {topk_ids.dtype} {tuple(topk_ids.shape)}")
    T = topk_ids.shape[0]
    if topk_w.dtype != torch.float32 or tuple(topk_w.shape) != (T, top_k):
        raise ValueError(f"topk_w must be float32 [{T}, {top_k}], got {topk_w.dtype} {tuple(topk_w.shape)}")
    if out.dtype != torch.float32 or tuple(out.shape) != (T, H):
        raise ValueError(f"out must be float32 [{T}, {H}], got {out.dtype} {tuple(out.shape)}")
    want_es = 4 if ad == MOE_F32 else 2
    if x.element_size() != want_es or x.dim() != 2 or tuple(x.shape) != (T, H):
        raise ValueError(f"x must be [{T}, {H}] with {want_es}-byte elements for adtype {adtype!r}, "
                         f"got {x.dtype} {tuple(x.shape)}")
    need = E * blob_bytes(wd, H, I)
    if _nbytes(experts) < need:
        raise ValueError(f"experts holds {_nbytes(experts)} bytes; E = {E} blobs need {need}")
    devs = {t.device for t in (experts, x, topk_ids, topk_w, out)}
    if len(devs) != 1 or next(iter(devs)).type != "cuda":
        raise ValueError(f"experts, x, topk_ids, topk_w and out must be on one CUDA device, got {sorted(map(str, devs))}")
    return T


def ffn_noalloc(experts, x, topk_ids, topk_w, out, *, E, H, I, top_k, wdtype, adtype, stream=None):
    """moe_layer_ffn_noalloc: all-resident expert SwiGLU + combine that allocates no GPU memory.

    For callers that may not allocate: every intermediate lives in the
    library's fixed device scratch array.  experts: the layer's E blobs back to
    back on the device.  Calls that overlap on the GPU share that scratch and
    race; order them on one stream.  Arguments whose sizes, dtypes or devices
    do not match E, H, I, top_k and the dtypes raise ValueError before the call.
    """
    T = _check_noalloc_args(experts, x, topk_ids, topk_w, out, E, H, I, top_k, wdtype, adtype)
    _check(load_library().moe_layer_ffn_noalloc(E, H, I, top_k, DTYPES.get(wdtype, wdtype),
                                                DTYPES.get(adtype, adtype), _ptr(experts), T, _ptr(x),
                                                _ptr(topk_ids), _ptr(topk_w), _ptr(out), _stream(stream)))
