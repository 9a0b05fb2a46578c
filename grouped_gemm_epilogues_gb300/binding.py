"""Thin ctypes binding of libgge.so (include/gge.h).

Argument marshalling only: torch tensors are turned into the C structs
(device pointer, dtype code, extents, element strides) and handed to the C
entry points of the same names; every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no fallback: if the library cannot be loaded, ``load()``
raises.
"""

import ctypes
import os
import threading

import torch

from . import build as _build

c_i32, c_i64, c_u32, c_u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64

DTYPE = {torch.bfloat16: 0, torch.float16: 1, torch.float8_e4m3fn: 2, torch.float8_e5m2: 3,
         torch.float32: 4}
ACT = {"none": 0, None: 0, "relu": 1, "gelu_tanh": 2, "gelu_tanh_approx": 2, "silu": 3,
       "relu_sq": 4}
STATUS = {0: "GGE_OK", 1: "GGE_ERR_INVALID_ARG", 2: "GGE_ERR_UNSUPPORTED",
          3: "GGE_ERR_ALIGNMENT", 4: "GGE_ERR_WORKSPACE", 5: "GGE_ERR_CUDA",
          6: "GGE_ERR_TIMEOUT", 7: "GGE_ERR_INDEX_RANGE"}


class GgeTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", c_i32), ("reserved", c_i32),
                ("rows", c_i64), ("cols", c_i64), ("batch", c_i64),
                ("stride_row", c_i64), ("stride_col", c_i64), ("stride_batch", c_i64)]


class GgeConfig(ctypes.Structure):
    _fields_ = [("tile_n", c_i32), ("num_ctas", c_i32), ("raster_band", c_i32),
                ("stages", c_i32), ("flags", c_i32), ("cta_group", c_i32),
                ("tile_counts", ctypes.c_void_p), ("timeout_ns", c_u64),
                ("batch_idx_permute", ctypes.c_void_p)]


class GgeGemmArgs(ctypes.Structure):
    _fields_ = [("A", GgeTensor), ("B", GgeTensor),
                ("C", ctypes.POINTER(GgeTensor)), ("D", ctypes.POINTER(GgeTensor)),
                ("PostAct", ctypes.POINTER(GgeTensor)),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("alpha_dev", ctypes.c_void_p), ("beta_dev", ctypes.c_void_p),
                ("act", c_i32), ("reserved", c_i32), ("config", ctypes.POINTER(GgeConfig))]


class GgePlanInfo(ctypes.Structure):
    _fields_ = [("tile_m", c_i32), ("tile_n", c_i32), ("tile_k", c_i32), ("stages", c_i32),
                ("num_tiles", c_i32), ("grid", c_i32), ("threads", c_i32),
                ("smem_bytes", c_i32), ("raster_band", c_i32), ("cta_group", c_i32),
                ("raster_along_n", c_i32), ("tail_tiles", c_i32), ("tail_splits", c_i32)]


# every function include/gge.h declares, with its ctypes signature
_SIGNATURES = {
    "gge_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(GgeGemmArgs), c_i32]),
    "gge_workspace_size_varlen_k": (ctypes.c_size_t, [ctypes.POINTER(GgeGemmArgs), c_i32]),
    "gge_gemm": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p, ctypes.c_size_t,
                         ctypes.c_void_p]),
    "gge_gemm_act": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p, ctypes.c_size_t,
                             ctypes.c_void_p]),
    "gge_gemm_varlen_m": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p, c_i32,
                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gge_gemm_varlen_k": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p, c_i32,
                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gge_gemm_gather_k": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p, ctypes.c_void_p,
                                  c_i32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gge_gemm_gather_a": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p, ctypes.c_void_p,
                                  c_i32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gge_gemm_dact": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p, ctypes.c_size_t,
                              ctypes.c_void_p]),
    "gge_gemm_act_static_scratch": (c_i32, [ctypes.POINTER(GgeGemmArgs), ctypes.c_void_p]),
    "gge_read_device_status": (c_i32, [ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.POINTER(c_i32)]),
    "gge_read_static_scratch_status": (c_i32, [ctypes.c_void_p, ctypes.POINTER(c_i32)]),
    "gge_status_string": (ctypes.c_char_p, [c_i32]),
    "gge_fastdivmod_params": (None, [c_i32, ctypes.POINTER(c_u32), ctypes.POINTER(c_u32)]),
    "gge_fastdivmod_div": (c_i32, [c_i32, c_i32]),
    "gge_schedule_map": (c_i32, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                 ctypes.POINTER(c_i32)]),
    "gge_plan": (c_i32, [ctypes.POINTER(GgeGemmArgs), c_i32, c_i32, ctypes.POINTER(GgePlanInfo)]),
    "gge_version": (ctypes.c_char_p, []),
    "gge_tune_candidates": (c_i32, [ctypes.POINTER(GgeGemmArgs), c_i32, c_i32,
                                    ctypes.POINTER(GgeConfig), c_i32]),
    "gge_autotune": (c_i32, [ctypes.POINTER(GgeGemmArgs), c_i32, ctypes.c_void_p, ctypes.c_void_p,
                             c_i32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, c_i32,
                             ctypes.POINTER(GgeConfig), ctypes.POINTER(ctypes.c_float)]),
    "gge_tuned_config": (c_i32, [ctypes.POINTER(GgeGemmArgs), c_i32, c_i32,
                                 ctypes.POINTER(GgeConfig)]),
}

_lib = None
_lock = threading.Lock()


class GgeError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{where}: {self.name}")


def load(path: str = None, build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgge.so (building it in-tree first if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise FileNotFoundError(path)
            _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ---------------------------------------------------------------- marshalling

def view(t: torch.Tensor, kind: str) -> GgeTensor:
    """C view of a torch tensor.  kind: 'mk' (A), 'nk' (B) or 'mn' (C/D/PostAct);
    2-D tensors are one batch, 3-D tensors are (batch, rows, cols)."""
    if t.dim() == 2:
        rows, cols = t.shape
        batch, sr, sc, sb = 1, t.stride(0), t.stride(1), t.numel()
    elif t.dim() == 3:
        batch, rows, cols = t.shape
        sb, sr, sc = t.stride()
    else:
        raise ValueError(f"{kind}: expected a 2-D or 3-D tensor")
    if t.dtype not in DTYPE:
        raise TypeError(f"{kind}: unsupported dtype {t.dtype}")
    return GgeTensor(ctypes.c_void_p(t.data_ptr()), DTYPE[t.dtype], 0, rows, cols, batch,
                     sr, sc, sb)


_workspaces = {}


def workspace(device=None, nbytes: int = 256) -> torch.Tensor:
    """The per-device workspace (zeroed when made), at least ``nbytes`` long.
    Growing it keeps the status words (the first 256 bytes) of the old one."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    ws = _workspaces.get(dev.index)
    if ws is None or ws.numel() < nbytes:
        new = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        if ws is not None:
            new[:256].copy_(ws[:256])
        ws = new
        _workspaces[dev.index] = ws
    return ws


def new_workspace(device=None, nbytes: int = 32 << 20) -> torch.Tensor:
    """A zeroed workspace of its own, for calls that may run at the same time on
    different streams: each such stream passes its own (``workspace=``) to the
    entry points, since by default every call on a device shares the one that
    ``workspace()`` keeps (its status words, scheduler counters and split tickets)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=dev)


_shared_workspace = workspace


def _ws(device, need, given):
    """The caller's workspace (checked), or the shared per-device one."""
    if given is None:
        return _shared_workspace(device, need)
    if given.dtype != torch.uint8 or given.device != device or not given.is_contiguous():
        raise ValueError("workspace: a contiguous uint8 tensor on the outputs' device")
    return given


# gge_config.flags bits (include/gge.h)
FLAGS = {
    "tile_counts": 1,          # count tile visits into tile_counts
    "test_drop_acc_full": 2,   # test hook: the epilogue's accumulator wait runs out
    "dynamic_sched": 4,        # tiles claimed from a counter in the workspace
    "direct_stores": 8,        # epilogue stores without shared-memory staging
    "no_split": 32,            # never split the last wave along K
    "raster_n": 128,           # raster bands of n-tiles
    "clc_sched": 256,          # cluster launch control: steal the tiles of unlaunched clusters
    "swap_ab": 512,            # compute D^T = B A^T (outputs stored transposed by the kernel)
    "k_serpentine": 1024,      # odd waves walk K backwards (L2 reuse across waves)
}
RESERVED_FLAGS = 16 | 64       # a call that sets one of these is rejected


def make_config(tile_n=0, num_ctas=0, raster_band=0, stages=0, flags=0, tile_counts=None,
                timeout_ns=0, cta_group=0, batch_idx_permute=None):
    """batch_idx_permute: None or a device int32 tensor [L] (a permutation of 0..L-1)."""
    return GgeConfig(tile_n, num_ctas, raster_band, stages, flags, cta_group,
                     ctypes.c_void_p(tile_counts.data_ptr()) if tile_counts is not None else None,
                     timeout_ns,
                     ctypes.c_void_p(batch_idx_permute.data_ptr())
                     if batch_idx_permute is not None else None)


def make_args(A, B, C=None, D=None, PostAct=None, alpha=1.0, beta=1.0, act="none",
              alpha_dev=None, beta_dev=None, config=None, a_kind="mk"):
    keep = []

    def opt(t):
        if t is None:
            return None
        v = view(t, "mn")
        keep.append(v)
        return ctypes.pointer(v)

    args = GgeGemmArgs()
    args.A = view(A, a_kind)
    args.B = view(B, "nk")
    args.C, args.D, args.PostAct = opt(C), opt(D), opt(PostAct)
    args.alpha, args.beta = float(alpha), float(beta)
    args.alpha_dev = ctypes.c_void_p(alpha_dev.data_ptr()) if alpha_dev is not None else None
    args.beta_dev = ctypes.c_void_p(beta_dev.data_ptr()) if beta_dev is not None else None
    args.act = ACT[act]
    args.config = ctypes.pointer(config) if config is not None else None
    args._keep = (keep, config)
    return args


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check(code, where):
    if code != 0:
        raise GgeError(code, where)


# ------------------------------------------------------------- entry points

def gge_gemm(A, B, D, C=None, alpha=1.0, beta=1.0, alpha_dev=None, beta_dev=None, config=None,
             workspace=None):
    """D = alpha * A @ B^T + beta * C.  A (L,M,K)/(M,K), B (L,N,K)/(N,K), D (L,M,N)/(M,N).
    workspace: optional buffer of the caller's (see new_workspace)."""
    lib = load()
    args = make_args(A, B, C=C, D=D, alpha=alpha, beta=beta, alpha_dev=alpha_dev,
                     beta_dev=beta_dev, config=config)
    ws = _ws(D.device, lib.gge_workspace_size(ctypes.byref(args), 0), workspace)
    _check(lib.gge_gemm(ctypes.byref(args), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                        _stream(D)), "gge_gemm")


def gge_gemm_act(A, B, PostAct, act, D=None, C=None, alpha=1.0, beta=1.0, alpha_dev=None,
                 beta_dev=None, config=None, workspace=None):
    """D (optional) and PostAct = act(alpha * A @ B^T + beta * C)."""
    lib = load()
    args = make_args(A, B, C=C, D=D, PostAct=PostAct, alpha=alpha, beta=beta, act=act,
                     alpha_dev=alpha_dev, beta_dev=beta_dev, config=config)
    ws = _ws(PostAct.device, lib.gge_workspace_size(ctypes.byref(args), 0), workspace)
    _check(lib.gge_gemm_act(ctypes.byref(args), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                            _stream(PostAct)), "gge_gemm_act")


def gge_gemm_dact(A, B, PreAct, D, act, PostAct=None, config=None, workspace=None):
    """Backward activation epilogue: D = act'(PreAct) * (A @ B^T), PostAct = act(PreAct)."""
    lib = load()
    args = make_args(A, B, C=PreAct, D=D, PostAct=PostAct, act=act, config=config)
    ws = _ws(D.device, lib.gge_workspace_size(ctypes.byref(args), 0), workspace)
    _check(lib.gge_gemm_dact(ctypes.byref(args), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                             _stream(D)), "gge_gemm_dact")


def gge_gemm_act_static_scratch(A, B, PostAct, act, D=None, C=None, alpha=1.0, beta=1.0,
                                config=None):
    """gge_gemm_act for callers that cannot allocate: no workspace argument, the
    library's own fixed scratch area is used (see include/gge.h)."""
    lib = load()
    args = make_args(A, B, C=C, D=D, PostAct=PostAct, alpha=alpha, beta=beta, act=act,
                     config=config)
    _check(lib.gge_gemm_act_static_scratch(ctypes.byref(args), _stream(PostAct)),
           "gge_gemm_act_static_scratch")


def gge_gemm_varlen_m(A, B, cu_seqlens_m, D=None, PostAct=None, act="none", C=None, alpha=1.0,
                      beta=1.0, config=None, workspace=None):
    """Varlen-M grouped GEMM: A (total_M, K), B (G, N, K), cu_seqlens_m int32 (G+1,) on device."""
    lib = load()
    out = D if D is not None else PostAct
    args = make_args(A, B, C=C, D=D, PostAct=PostAct, alpha=alpha, beta=beta, act=act,
                     config=config)
    ws = _ws(out.device, 256, workspace)
    G = cu_seqlens_m.numel() - 1
    _check(lib.gge_gemm_varlen_m(ctypes.byref(args), ctypes.c_void_p(cu_seqlens_m.data_ptr()), G,
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(out)),
           "gge_gemm_varlen_m")


def gge_gemm_varlen_k(A, B, cu_seqlens_k, D=None, PostAct=None, act="none", C=None, alpha=1.0,
                      beta=1.0, config=None, workspace=None):
    """Varlen-K grouped GEMM: A (M, total_K), B (N, total_K), cu_seqlens_k int32 (G+1,) on
    device; C / D / PostAct (G, M, N).  Group g contracts K columns cu[g] .. cu[g+1]-1."""
    lib = load()
    out = D if D is not None else PostAct
    args = make_args(A, B, C=C, D=D, PostAct=PostAct, alpha=alpha, beta=beta, act=act,
                     config=config)
    G = cu_seqlens_k.numel() - 1
    need = lib.gge_workspace_size_varlen_k(ctypes.byref(args), G)
    ws = _ws(out.device, need, workspace)
    _check(lib.gge_gemm_varlen_k(ctypes.byref(args), ctypes.c_void_p(cu_seqlens_k.data_ptr()), G,
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(out)),
           "gge_gemm_varlen_k")


def gge_gemm_gather_k(A_src, B, a_idx, cu_seqlens_k, D=None, PostAct=None, act="none", C=None,
                      alpha=1.0, beta=1.0, config=None, workspace=None):
    """Gather-K: varlen-K GEMM whose A column k is A_src[:, a_idx[k]].  A_src (M, K_src)
    M-major (e.g. X.t() of a row-major X [K_src, M]), B (N, total_K), a_idx int32
    (total_K,), cu_seqlens_k int32 (G+1,); C / D / PostAct (G, M, N)."""
    lib = load()
    out = D if D is not None else PostAct
    args = make_args(A_src, B, C=C, D=D, PostAct=PostAct, alpha=alpha, beta=beta, act=act,
                     config=config)
    G = cu_seqlens_k.numel() - 1
    ws = _ws(out.device, lib.gge_workspace_size_varlen_k(ctypes.byref(args), G), workspace)
    _check(lib.gge_gemm_gather_k(ctypes.byref(args), ctypes.c_void_p(a_idx.data_ptr()),
                                 ctypes.c_void_p(cu_seqlens_k.data_ptr()), G,
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(out)),
           "gge_gemm_gather_k")


def gge_gemm_gather_a(A_src, B, a_idx, cu_seqlens_m=None, D=None, PostAct=None, act="none",
                      C=None, alpha=1.0, beta=1.0, config=None, workspace=None):
    """Gather-A GEMM: effective A row r = A_src[a_idx[r]]; varlen-M when cu_seqlens_m is given."""
    lib = load()
    out = D if D is not None else PostAct
    args = make_args(A_src, B, C=C, D=D, PostAct=PostAct, alpha=alpha, beta=beta, act=act,
                     config=config)
    ws = _ws(out.device, 256, workspace)
    G = cu_seqlens_m.numel() - 1 if cu_seqlens_m is not None else 0
    cu = ctypes.c_void_p(cu_seqlens_m.data_ptr()) if cu_seqlens_m is not None else None
    _check(lib.gge_gemm_gather_a(ctypes.byref(args), ctypes.c_void_p(a_idx.data_ptr()), cu, G,
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(out)),
           "gge_gemm_gather_a")


def gge_read_static_scratch_status(device=None):
    """Synchronise the current stream and return (status_name, where, tile) that
    gge_gemm_act_static_scratch calls recorded in the library's area; clears it."""
    lib = load()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    detail = (c_i32 * 2)()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    code = lib.gge_read_static_scratch_status(stream, detail)
    return STATUS.get(code, str(code)), detail[0], detail[1]


def gge_read_device_status(device=None, workspace=None):
    """Synchronise the current stream and return (status_name, where, tile) recorded in
    the shared per-device workspace (or in ``workspace``, a caller's); clears it."""
    lib = load()
    ws = workspace if workspace is not None else _shared_workspace(device)
    detail = (c_i32 * 2)()
    code = lib.gge_read_device_status(ctypes.c_void_p(ws.data_ptr()), _stream(ws), detail)
    return STATUS.get(code, str(code)), detail[0], detail[1]


FORM = {"default": 0, "gather_a": 1, "varlen_k": 2, "gather_k": 3}


def gge_plan(A, B, C=None, D=None, PostAct=None, act="none", num_groups=0, gather=False,
             config=None, form=None):
    """The launch plan; form: 'default' (plain / varlen-M), 'gather_a' or 'varlen_k'."""
    lib = load()
    args = make_args(A, B, C=C, D=D, PostAct=PostAct, act=act, config=config)
    info = GgePlanInfo()
    f = FORM[form] if form is not None else (1 if gather else 0)
    code = lib.gge_plan(ctypes.byref(args), num_groups, f, ctypes.byref(info))
    _check(code, "gge_plan")
    return {k: getattr(info, k) for k, _ in GgePlanInfo._fields_}


# ------------------------------------------------------------------ autotuning

OP = {"gemm": 0, "dact": 1, "varlen_m": 2, "gather_a": 3, "varlen_k": 4, "gather_k": 5}
_CFG_KEYS = ("tile_n", "num_ctas", "raster_band", "stages", "flags", "cta_group")


def config_dict(c: GgeConfig) -> dict:
    return {k: getattr(c, k) for k in _CFG_KEYS}


def _tune_args(op, A, B, C, D, PostAct, act, alpha, beta, config):
    if op == "dact":   # the backward epilogue reads the pre-activation from C
        return make_args(A, B, C=C, D=D, PostAct=PostAct, act=act, config=config)
    return make_args(A, B, C=C, D=D, PostAct=PostAct, alpha=alpha, beta=beta, act=act,
                     config=config)


def gge_tune_candidates(op, A, B, C=None, D=None, PostAct=None, act="none", num_groups=0,
                        config=None):
    """The launch configurations gge_autotune would time for this problem (host only)."""
    lib = load()
    args = _tune_args(op, A, B, C, D, PostAct, act, 1.0, 1.0, config)
    out = (GgeConfig * 64)()
    n = lib.gge_tune_candidates(ctypes.byref(args), OP[op], num_groups, out, 64)
    return [config_dict(out[i]) for i in range(min(n, 64))]


def gge_autotune(op, A, B, idx=None, cu=None, C=None, D=None, PostAct=None, act="none",
                 alpha=1.0, beta=1.0, reps=10, config=None):
    """Time every candidate launch shape of `op` on the current stream and return
    (best config as a dict, its mean time in ms).  The outputs hold the result."""
    lib = load()
    out = D if D is not None else PostAct
    args = _tune_args(op, A, B, C, D, PostAct, act, alpha, beta, config)
    G = cu.numel() - 1 if cu is not None else 0
    if op in ("varlen_k", "gather_k"):
        need = lib.gge_workspace_size_varlen_k(ctypes.byref(args), G)
    else:
        need = lib.gge_workspace_size(ctypes.byref(args), G)
    ws = workspace(out.device, need)
    best = GgeConfig()
    ms = ctypes.c_float()
    code = lib.gge_autotune(ctypes.byref(args), OP[op],
                            ctypes.c_void_p(idx.data_ptr()) if idx is not None else None,
                            ctypes.c_void_p(cu.data_ptr()) if cu is not None else None, G,
                            ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(out), reps,
                            ctypes.byref(best), ctypes.byref(ms))
    _check(code, "gge_autotune")
    return config_dict(best), ms.value


def gge_tuned_config(op, A, B, C=None, D=None, PostAct=None, act="none", num_groups=0,
                     config=None):
    """The configuration gge_autotune stored for a problem of this key, or None."""
    lib = load()
    args = _tune_args(op, A, B, C, D, PostAct, act, 1.0, 1.0, config)
    c = GgeConfig()
    if lib.gge_tuned_config(ctypes.byref(args), OP[op], num_groups, ctypes.byref(c)) != 0:
        return None
    return config_dict(c)
