"""ctypes binding of the C ABI in ``include/cs_chain.h``.

Argument marshalling only: tensors become device pointers, the current torch
stream becomes a ``cudaStream_t``; every step of the chain runs in the CUDA
library.  If the library is missing, importing this module raises ImportError:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))


def library_path(environ=os.environ) -> str:
    """The build this process loads.  A process that shares a node with other
    GPUs' ranks (WORLD_SIZE > 1, as torchrun sets it) loads the replica build,
    which contains no TMA cluster-multicast load; CS_CHAIN_LIBRARY=full|nomc
    overrides the choice."""
    want = environ.get("CS_CHAIN_LIBRARY", "")
    if want not in ("", "full", "nomc"):
        raise ImportError(f"CS_CHAIN_LIBRARY={want!r}: expected 'full' or 'nomc'")
    ws = environ.get("WORLD_SIZE", "1")
    nomc = want == "nomc" or (want == "" and ws.isdigit() and int(ws) > 1)
    return os.path.join(PKG, "_lib", "libcs_chain_nomc.so" if nomc else "libcs_chain.so")


LIB_PATH = library_path()

# cs_status
CS_OK = 0
CS_ERR_INVALID_ARG = 1
CS_ERR_UNSUPPORTED = 2
CS_ERR_CUDA = 3
CS_ERR_TIMEOUT = 4
CS_ERR_OOM = 5
CS_ERR_WATCHDOG = 6
CS_ERR_NEEDS_RESET = 7
STATUS_NAMES = {0: "CS_OK", 1: "CS_ERR_INVALID_ARG", 2: "CS_ERR_UNSUPPORTED", 3: "CS_ERR_CUDA",
                4: "CS_ERR_TIMEOUT", 5: "CS_ERR_OOM", 6: "CS_ERR_WATCHDOG", 7: "CS_ERR_NEEDS_RESET"}
# enums
CS_F16, CS_BF16 = 0, 1
CS_CHAIN_MLP_GELU, CS_CHAIN_MLP_SWIGLU, CS_CHAIN_ATTN = 0, 1, 2
CS_SYNC_AUTO, CS_SYNC_TILE, CS_SYNC_ROW, CS_SYNC_STRIDED, CS_SYNC_STREAM = -1, 0, 1, 2, 3
CS_WEIGHTS_KN, CS_WEIGHTS_NK = 0, 1
POLICIES = {"auto": CS_SYNC_AUTO, "tile": CS_SYNC_TILE, "row": CS_SYNC_ROW, "strided": CS_SYNC_STRIDED,
            "stream": CS_SYNC_STREAM}
POLICY_NAMES = {v: k for k, v in POLICIES.items()}
# the tuning table measured on this package's target GPU (written by the tuner,
# consumer_gemm_chain_gb300.tune); cs_tune_load() reads it
TUNE_TABLE = os.path.join(PKG, "tuning", "gb300.json")
KINDS = {"gelu": CS_CHAIN_MLP_GELU, "swiglu": CS_CHAIN_MLP_SWIGLU, "attn": CS_CHAIN_ATTN}

EXPORTED = (
    "cs_chain_desc_init", "cs_chain_plan", "cs_chain_destroy", "cs_mlp_forward", "cs_mlp_forward_host",
    "cs_chain_host_join", "cs_attn_chain_forward",
    "cs_chain_forward_stage", "cs_chain_status", "cs_chain_reset", "cs_last_error_string", "cs_chain_query",
    "cs_schedule_build", "cs_chain_debug_read_sems", "cs_chain_debug_set_delays", "cs_chain_debug_skip_release",
    "cs_chain_debug_copy_intermediate", "cs_chain_debug_trace", "cs_chain_debug_read_trace", "cs_abi_version",
    "cs_mlp_forward_noalloc", "cs_noalloc_status", "cs_tune_load", "cs_tune_clear", "cs_tune_size",
    "cs_tune_match", "cs_chain_plan_info", "cs_library_features", "cs_chain_debug_poison_intermediate",
    "cs_chain_debug_set_epoch",
)
CS_FEATURE_CLUSTER_MULTICAST = 1


class cs_chain_desc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("M", ctypes.c_int), ("H", ctypes.c_int), ("F", ctypes.c_int),
                ("dtype", ctypes.c_int), ("policy", ctypes.c_int), ("weight_layout", ctypes.c_int),
                ("stride", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("num_sms", ctypes.c_int), ("lag", ctypes.c_int), ("group_m", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("tile_m", ctypes.c_int), ("split_k", ctypes.c_int),
                ("prefetch", ctypes.c_int), ("raster", ctypes.c_int), ("pdl", ctypes.c_int),
                ("tuned", ctypes.c_int), ("out_release", ctypes.c_int), ("spin_timeout_ns", ctypes.c_ulonglong),
                ("sk_tiles", ctypes.c_int), ("sk_units", ctypes.c_int), ("kv_chunk", ctypes.c_int),
                ("split_k_first", ctypes.c_int)]


class cs_mlp_args(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("W1", ctypes.c_void_p), ("b1", ctypes.c_void_p), ("Wg", ctypes.c_void_p),
                ("Wu", ctypes.c_void_p), ("W2", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


class cs_attn_args(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("Wqkv", ctypes.c_void_p), ("Wo", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


class cs_chain_info(ctypes.Structure):
    _fields_ = [("stages", ctypes.c_int), ("m_tiles", ctypes.c_int), ("n_tiles", ctypes.c_int * 3),
                ("units", ctypes.c_int * 3), ("n_units", ctypes.c_int), ("num_sms", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("lag", ctypes.c_int), ("group_m", ctypes.c_int),
                ("tile_n", ctypes.c_int * 3), ("tile_m", ctypes.c_int), ("sched_units", ctypes.c_int * 3),
                ("split_k", ctypes.c_int * 3),
                ("stride", ctypes.c_int),
                ("intermediate", ctypes.c_void_p * 2), ("sem_words", ctypes.c_size_t * 2),
                ("policy", ctypes.c_int), ("tuned_entry", ctypes.c_int),
                ("out_tile_sems", ctypes.c_void_p), ("out_row_sems", ctypes.c_void_p), ("out_sem_words", ctypes.c_size_t),
                ("sk_tiles", ctypes.c_int), ("sk_units", ctypes.c_int), ("sk_q", ctypes.c_int),
                ("workers", ctypes.c_int), ("kv_chunk", ctypes.c_int), ("raster", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"the CUDA library {LIB_PATH} is not built; run consumer_gemm_chain_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    V, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "cs_chain_desc_init": (I, [ctypes.POINTER(cs_chain_desc)]),
        "cs_chain_plan": (I, [ctypes.POINTER(cs_chain_desc), ctypes.POINTER(V)]),
        "cs_chain_destroy": (I, [V]),
        "cs_mlp_forward": (I, [V, ctypes.POINTER(cs_mlp_args), V]),
        "cs_mlp_forward_host": (I, [V, ctypes.POINTER(cs_mlp_args), V]),
        "cs_chain_host_join": (I, [V, V]),
        "cs_attn_chain_forward": (I, [V, ctypes.POINTER(cs_attn_args), V]),
        "cs_chain_forward_stage": (I, [V, V, I, V]),
        "cs_chain_status": (I, [V]),
        "cs_chain_reset": (I, [V]),
        "cs_last_error_string": (ctypes.c_char_p, []),
        "cs_chain_query": (I, [V, ctypes.POINTER(cs_chain_info)]),
        "cs_schedule_build": (I, [ctypes.POINTER(cs_chain_desc), I, ctypes.POINTER(ctypes.c_uint32), S,
                                  ctypes.POINTER(S)]),
        "cs_chain_debug_read_sems": (I, [V, I, ctypes.POINTER(ctypes.c_uint32), S, ctypes.POINTER(ctypes.c_uint32)]),
        "cs_chain_debug_set_delays": (I, [V, I, ctypes.POINTER(ctypes.c_uint32), S]),
        "cs_chain_debug_skip_release": (I, [V, I, I]),
        "cs_chain_debug_copy_intermediate": (I, [V, I, V, S]),
        "cs_chain_debug_trace": (I, [V, I]),
        "cs_chain_debug_read_trace": (I, [V, ctypes.POINTER(ctypes.c_uint64), S, ctypes.POINTER(S)]),
        "cs_abi_version": (I, []),
        "cs_mlp_forward_noalloc": (I, [ctypes.POINTER(cs_chain_desc), ctypes.POINTER(cs_mlp_args), V]),
        "cs_noalloc_status": (I, []),
        "cs_tune_load": (I, [ctypes.c_char_p, ctypes.POINTER(I)]),
        "cs_tune_clear": (I, []),
        "cs_tune_size": (I, []),
        "cs_tune_match": (I, [ctypes.POINTER(cs_chain_desc), I, ctypes.POINTER(I), ctypes.POINTER(cs_chain_desc)]),
        "cs_chain_plan_info": (I, [ctypes.POINTER(cs_chain_desc), I, ctypes.POINTER(cs_chain_info)]),
        "cs_library_features": (I, []),
        "cs_chain_debug_poison_intermediate": (I, [V, I, V]),
        "cs_chain_debug_set_epoch": (I, [V, ctypes.c_uint32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


class CSError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib.cs_last_error_string().decode(errors="replace")
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}: {msg}")


def _check(status: int, what: str) -> None:
    if status != CS_OK:
        raise CSError(status, what)


def cs_abi_version() -> int:
    return _lib.cs_abi_version()


def cs_last_error_string() -> str:
    return _lib.cs_last_error_string().decode(errors="replace")


def cs_chain_desc_init(**fields) -> cs_chain_desc:
    """A desc with the library defaults, then ``fields`` applied (names as in the C struct;
    ``kind``/``policy`` also accept "gelu"/"swiglu"/"attn" and "tile"/"row"/"strided"/"stream";
    ``dtype`` accepts torch dtypes)."""
    d = cs_chain_desc()
    _check(_lib.cs_chain_desc_init(ctypes.byref(d)), "cs_chain_desc_init")
    for k, v in fields.items():
        if k == "kind" and isinstance(v, str):
            v = KINDS[v]
        elif k == "policy" and isinstance(v, str):
            v = POLICIES[v]
        elif k == "dtype" and not isinstance(v, int):
            v = _dtype_code(v)
        elif k == "weight_layout" and isinstance(v, str):
            v = {"kn": CS_WEIGHTS_KN, "nk": CS_WEIGHTS_NK}[v.lower()]
        setattr(d, k, v)
    return d


def _dtype_code(dt) -> int:
    import torch
    if dt == torch.float16:
        return CS_F16
    if dt == torch.bfloat16:
        return CS_BF16
    raise ValueError(f"unsupported dtype {dt}")


class Plan:
    """Handle of a plan made by :func:`cs_chain_plan` (destroy with :func:`cs_chain_destroy`)."""

    def __init__(self, handle: int, desc: cs_chain_desc):
        self.handle = handle
        self.desc = desc

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        cs_chain_destroy(self)

    def __del__(self):
        try:
            cs_chain_destroy(self)
        except Exception:
            pass


def cs_chain_plan(desc: cs_chain_desc) -> Plan:
    h = ctypes.c_void_p()
    _check(_lib.cs_chain_plan(ctypes.byref(desc), ctypes.byref(h)), "cs_chain_plan")
    d = cs_chain_desc()
    ctypes.memmove(ctypes.byref(d), ctypes.byref(desc), ctypes.sizeof(desc))
    return Plan(h.value, d)


def cs_chain_destroy(plan: Plan) -> None:
    if plan is not None and plan.handle:
        h, plan.handle = plan.handle, None
        _check(_lib.cs_chain_destroy(h), "cs_chain_destroy")


def _stream_ptr(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, shape, dtype, name, host=False):
    """Device (host=True: host) pointer of tensor t after checking shape/dtype/contiguity/device."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if host and t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not host and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, the plan uses {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _torch_dtype(desc):
    import torch
    return torch.bfloat16 if desc.dtype == CS_BF16 else torch.float16


def _wshape(desc, K, N):
    return (K, N) if desc.weight_layout == CS_WEIGHTS_KN else (N, K)


def _mlp_args(plan: Plan, X, W1=None, b1=None, W2=None, Y=None, Wg=None, Wu=None) -> cs_mlp_args:
    d = plan.desc
    dt = _torch_dtype(d)
    M, H, F = d.M, d.H, d.F
    a = cs_mlp_args()
    a.X = _ptr(X, (M, H), dt, "X")
    a.W1 = _ptr(W1, _wshape(d, H, F), dt, "W1")
    a.b1 = _ptr(b1, (F,), dt, "b1")
    a.Wg = _ptr(Wg, _wshape(d, H, F), dt, "Wg")
    a.Wu = _ptr(Wu, _wshape(d, H, F), dt, "Wu")
    a.W2 = _ptr(W2, _wshape(d, F, H), dt, "W2")
    a.Y = _ptr(Y, (M, H), dt, "Y")
    return a


def cs_mlp_forward(plan: Plan, X, W1=None, b1=None, W2=None, Y=None, Wg=None, Wu=None, stream=None) -> None:
    """Enqueue Y = GeLU(X W1 + b1) W2 (or the SwiGLU chain with Wg, Wu, W2=Wd) on ``stream``."""
    a = _mlp_args(plan, X, W1, b1, W2, Y, Wg, Wu)
    _check(_lib.cs_mlp_forward(plan.handle, ctypes.byref(a), _stream_ptr(stream)), "cs_mlp_forward")


def cs_mlp_forward_host(plan: Plan, X, W1=None, b1=None, W2=None, Y=None, Wg=None, Wu=None, stream=None) -> None:
    """Like cs_mlp_forward with X and Y in host memory (CPU tensors, pinned for
    the copies to overlap the kernels); Y holds the result after
    cs_chain_host_join on a stream and a synchronisation of that stream."""
    d = plan.desc
    dt = _torch_dtype(d)
    a = _mlp_args(plan, None, W1, b1, W2, None, Wg, Wu)
    a.X = _ptr(X, (d.M, d.H), dt, "X", host=True)
    a.Y = _ptr(Y, (d.M, d.H), dt, "Y", host=True)
    _check(_lib.cs_mlp_forward_host(plan.handle, ctypes.byref(a), _stream_ptr(stream)), "cs_mlp_forward_host")


def cs_chain_host_join(plan: Plan, stream=None) -> None:
    """Make ``stream`` wait for every Y read-back of cs_mlp_forward_host so far."""
    _check(_lib.cs_chain_host_join(plan.handle, _stream_ptr(stream)), "cs_chain_host_join")


def _attn_args(plan: Plan, X, Wqkv, Wo, Y) -> cs_attn_args:
    d = plan.desc
    dt = _torch_dtype(d)
    a = cs_attn_args()
    a.X = _ptr(X, (d.M, d.H), dt, "X")
    a.Wqkv = _ptr(Wqkv, _wshape(d, d.H, 3 * d.F), dt, "Wqkv")
    a.Wo = _ptr(Wo, _wshape(d, d.F, d.H), dt, "Wo")
    a.Y = _ptr(Y, (d.M, d.H), dt, "Y")
    return a


def cs_attn_chain_forward(plan: Plan, X, Wqkv, Wo, Y, stream=None) -> None:
    """Enqueue QKV = X Wqkv -> causal attention per head -> Y = O Wo on ``stream``."""
    a = _attn_args(plan, X, Wqkv, Wo, Y)
    _check(_lib.cs_attn_chain_forward(plan.handle, ctypes.byref(a), _stream_ptr(stream)), "cs_attn_chain_forward")


def cs_chain_forward_stage(plan: Plan, stage: int, stream=None, **tensors) -> None:
    """Run one stage alone (no waits, no releases).  ``tensors`` as for the chain's forward."""
    if plan.desc.kind == CS_CHAIN_ATTN:
        a = _attn_args(plan, tensors.get("X"), tensors.get("Wqkv"), tensors.get("Wo"), tensors.get("Y"))
    else:
        a = _mlp_args(plan, **tensors)
    _check(_lib.cs_chain_forward_stage(plan.handle, ctypes.cast(ctypes.byref(a), ctypes.c_void_p), stage,
                                       _stream_ptr(stream)), "cs_chain_forward_stage")


def cs_chain_status(plan: Plan) -> int:
    """Device status of the plan's last forwards (after a stream sync): a cs_status code."""
    return _lib.cs_chain_status(plan.handle)


def cs_chain_reset(plan: Plan) -> None:
    _check(_lib.cs_chain_reset(plan.handle), "cs_chain_reset")


def cs_chain_query(plan: Plan) -> dict:
    i = cs_chain_info()
    _check(_lib.cs_chain_query(plan.handle, ctypes.byref(i)), "cs_chain_query")
    return _info_dict(i)


def cs_chain_plan_info(desc: cs_chain_desc, num_sms: int) -> dict:
    """The geometry a plan of ``desc`` would get on ``num_sms`` SMs (keys as
    cs_chain_query; pointers are None).  Needs no GPU."""
    i = cs_chain_info()
    _check(_lib.cs_chain_plan_info(ctypes.byref(desc), num_sms, ctypes.byref(i)), "cs_chain_plan_info")
    return _info_dict(i)


def cs_library_features() -> int:
    """Bit flags of the loaded build (CS_FEATURE_CLUSTER_MULTICAST)."""
    return _lib.cs_library_features()


def _info_dict(i: cs_chain_info) -> dict:
    return {"stages": i.stages, "m_tiles": i.m_tiles, "n_tiles": list(i.n_tiles), "units": list(i.units),
            "n_units": i.n_units, "num_sms": i.num_sms, "smem_bytes": i.smem_bytes, "lag": i.lag,
            "group_m": i.group_m, "tile_n": list(i.tile_n), "tile_m": i.tile_m,
            "sched_units": list(i.sched_units), "split_k": list(i.split_k),
            "stride": i.stride, "intermediate": [i.intermediate[0], i.intermediate[1]],
            "sem_words": [i.sem_words[0], i.sem_words[1]], "policy": POLICY_NAMES.get(i.policy, i.policy),
            "tuned_entry": i.tuned_entry, "out_tile_sems": i.out_tile_sems, "out_row_sems": i.out_row_sems,
            "out_sem_words": i.out_sem_words, "sk_tiles": i.sk_tiles, "sk_units": i.sk_units, "sk_q": i.sk_q,
            "workers": i.workers, "kv_chunk": i.kv_chunk, "raster": i.raster}


def cs_schedule_build(desc: cs_chain_desc, num_sms: int) -> list[int]:
    n = ctypes.c_size_t()
    _check(_lib.cs_schedule_build(ctypes.byref(desc), num_sms, None, 0, ctypes.byref(n)), "cs_schedule_build")
    buf = (ctypes.c_uint32 * max(1, n.value))()
    _check(_lib.cs_schedule_build(ctypes.byref(desc), num_sms, buf, n.value, ctypes.byref(n)), "cs_schedule_build")
    return list(buf[: n.value])


def cs_tune_load(path: str | None = None) -> int:
    """Replace the process-wide tuning table with a JSON file (default: the
    table measured for this package's target GPU); returns the entry count.
    Plans made afterwards take their auto fields from it (cs_chain_desc.tuned)."""
    n = ctypes.c_int()
    path = TUNE_TABLE if path is None else os.fspath(path)
    _check(_lib.cs_tune_load(path.encode(), ctypes.byref(n)), "cs_tune_load")
    return n.value


def cs_tune_clear() -> None:
    _check(_lib.cs_tune_clear(), "cs_tune_clear")


def cs_tune_size() -> int:
    return _lib.cs_tune_size()


def cs_tune_match(desc: cs_chain_desc, num_sms: int) -> tuple[int, cs_chain_desc]:
    """(index of the table entry a plan of ``desc`` on ``num_sms`` SMs applies, or -1;
    the desc as that plan runs it).  Needs no GPU."""
    e = ctypes.c_int()
    r = cs_chain_desc()
    _check(_lib.cs_tune_match(ctypes.byref(desc), num_sms, ctypes.byref(e), ctypes.byref(r)), "cs_tune_match")
    return e.value, r


def decode_unit(u: int) -> tuple[int, int, int, int]:
    """(stage, m_tile, n_tile, k_split) of a schedule entry."""
    return u >> 30, (u >> 14) & 0xFFF, u & 0x3FFF, (u >> 26) & 0xF


def cs_chain_debug_read_sems(plan: Plan, boundary: int):
    """(tile semaphores as a [m_tiles, n_tiles] list of lists, row counters, epoch)."""
    q = cs_chain_query(plan)
    sem_words = q["out_sem_words"] if boundary == q["stages"] - 1 else q["sem_words"][boundary]
    words = sem_words + q["m_tiles"]
    buf = (ctypes.c_uint32 * words)()
    ep = ctypes.c_uint32()
    _check(_lib.cs_chain_debug_read_sems(plan.handle, boundary, buf, words, ctypes.byref(ep)),
           "cs_chain_debug_read_sems")
    vals = list(buf)
    nt = q["n_tiles"][boundary]
    tiles = [vals[m * nt:(m + 1) * nt] for m in range(q["m_tiles"])]
    rows = vals[sem_words:]
    return tiles, rows, ep.value


def cs_chain_debug_set_delays(plan: Plan, stage: int, ns=None) -> None:
    if ns is None:
        _check(_lib.cs_chain_debug_set_delays(plan.handle, stage, None, 0), "cs_chain_debug_set_delays")
        return
    arr = (ctypes.c_uint32 * len(ns))(*[int(v) for v in ns])
    _check(_lib.cs_chain_debug_set_delays(plan.handle, stage, arr, len(ns)), "cs_chain_debug_set_delays")


def cs_chain_debug_skip_release(plan: Plan, stage: int, unit: int) -> None:
    _check(_lib.cs_chain_debug_skip_release(plan.handle, stage, unit), "cs_chain_debug_skip_release")


def cs_chain_debug_copy_intermediate(plan: Plan, which: int, out) -> None:
    """Copy plan-owned intermediate ``which`` into the CUDA tensor ``out`` (blocking)."""
    nbytes = out.numel() * out.element_size()
    _check(_lib.cs_chain_debug_copy_intermediate(plan.handle, which, out.data_ptr(), nbytes),
           "cs_chain_debug_copy_intermediate")


def cs_chain_debug_poison_intermediate(plan: Plan, which: int = -1, stream=None) -> None:
    """Enqueue a NaN fill of plan-owned scratch (0: H or QKV, 1: O, 2: split-K
    partial tiles, -1: all): a consumer that read before its producer released
    would then produce NaN."""
    _check(_lib.cs_chain_debug_poison_intermediate(plan.handle, which, _stream_ptr(stream)),
           "cs_chain_debug_poison_intermediate")


def cs_chain_debug_set_epoch(plan: Plan, epoch: int) -> None:
    """Set the epoch and every counter to their values after ``epoch`` forwards (mod 2^32)."""
    _check(_lib.cs_chain_debug_set_epoch(plan.handle, epoch & 0xFFFFFFFF), "cs_chain_debug_set_epoch")


def cs_chain_debug_trace(plan: Plan, enable: bool = True) -> None:
    """Record a per-unit timeline in every later forward (see cs_chain.h)."""
    _check(_lib.cs_chain_debug_trace(plan.handle, 1 if enable else 0), "cs_chain_debug_trace")


def cs_chain_debug_read_trace(plan: Plan) -> list[list[int]]:
    """Trace records (8 integers each) of the latest forward."""
    n = ctypes.c_size_t()
    _check(_lib.cs_chain_debug_read_trace(plan.handle, None, 0, ctypes.byref(n)), "cs_chain_debug_read_trace")
    buf = (ctypes.c_uint64 * (8 * max(1, n.value)))()
    _check(_lib.cs_chain_debug_read_trace(plan.handle, buf, n.value, ctypes.byref(n)), "cs_chain_debug_read_trace")
    vals = list(buf)
    return [vals[i * 8:(i + 1) * 8] for i in range(n.value)]


class _DescOnly:
    """Shape holder for the argument checks of calls that take a desc, not a plan."""

    def __init__(self, desc: cs_chain_desc):
        self.desc = desc


def cs_mlp_forward_noalloc(desc: cs_chain_desc, X, W1=None, b1=None, W2=None, Y=None, Wg=None, Wu=None,
                           stream=None) -> None:
    """The MLP chain without a plan and without any device allocation: for callers
    that may not call cudaMalloc (inside another framework's memory pool, or in
    loops where an allocation's implicit device synchronisation is not allowed).
    Scratch is a fixed 32 MiB array inside the library; calls that overlap on
    the GPU race.  See include/cs_chain.h."""
    a = _mlp_args(_DescOnly(desc), X, W1, b1, W2, Y, Wg, Wu)
    _check(_lib.cs_mlp_forward_noalloc(ctypes.byref(desc), ctypes.byref(a), _stream_ptr(stream)),
           "cs_mlp_forward_noalloc")


def cs_noalloc_status() -> int:
    """Device status of the last allocation-free forward on the current device (after a sync)."""
    return _lib.cs_noalloc_status()
