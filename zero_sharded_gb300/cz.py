"""ctypes binding of libcz (include/cz.h): argument marshalling only.

Every function keeps the C-ABI name.  Device buffers are passed as torch
tensors (their data pointers) or raw integers; host arrays are converted to
contiguous int64 buffers.  There is no fallback: if libcz.so is not built,
loading raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

from . import build as _build

CZ_OK = 0
CZ_ERR_INVALID = -1
CZ_ERR_CUDA = -2
CZ_ERR_NOMEM = -3
CZ_ERR_PLAN_MISMATCH = -4
CZ_ERR_TIMEOUT = -5
CZ_ERR_DEVICE_CHECK = -6
CZ_ERR_UNSUPPORTED = -7

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


class cz_step_opts(ctypes.Structure):
    _fields_ = [
        ("nesterov", ctypes.c_int32),
        ("eps", ctypes.c_float),
        ("a", ctypes.c_float),
        ("b", ctypes.c_float),
        ("c", ctypes.c_float),
        ("grad_is_bf16", ctypes.c_int32),
        ("param_bf16", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("debug_update_out", ctypes.c_void_p),
        ("lr_device", ctypes.c_void_p),
    ]


class CzError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        super().__init__(f"{fn} failed: {status} ({cz_status_string(status)})" + (f": {detail}" if detail else ""))
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the in-tree libcz.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libcz.so not built at {path}; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    sig = {
        "cz_make_buckets": (ctypes.c_int, [_i64p, ctypes.c_int64, ctypes.c_int64, _i64p, _i64p]),
        "cz_plan_partition": (ctypes.c_int, [_i64p, ctypes.c_int64, _i64p, ctypes.c_int64, ctypes.c_int32,
                                             ctypes.c_double, ctypes.POINTER(ctypes.c_void_p)]),
        "cz_plan_naive": (ctypes.c_int, [_i64p, ctypes.c_int64, _i64p, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.POINTER(ctypes.c_void_p)]),
        "cz_plan_partition_cost": (ctypes.c_int, [_i64p, _i64p, ctypes.c_int64, _i64p, ctypes.c_int64,
                                                  ctypes.c_int32, ctypes.c_double, ctypes.POINTER(ctypes.c_void_p)]),
        "cz_plan_rank_elems": (ctypes.c_int, [ctypes.c_void_p, _i64p]),
        "cz_plan_microgroups": (ctypes.c_int, [_i64p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, _i32p, _i32p,
                                               _i64p]),
        "cz_plan_free": (None, [ctypes.c_void_p]),
        "cz_plan_info": (ctypes.c_int, [ctypes.c_void_p, _i64p, _i64p, _i32p]),
        "cz_plan_owner": (ctypes.c_int, [ctypes.c_void_p, _i32p]),
        "cz_plan_cuts": (ctypes.c_int, [ctypes.c_void_p, _i64p, _i64p]),
        "cz_plan_rank_load": (ctypes.c_int, [ctypes.c_void_p, _i64p]),
        "cz_plan_metrics": (ctypes.c_int, [ctypes.c_void_p, _f64p, _f64p, _f64p]),
        "cz_step_opts_default": (None, [ctypes.POINTER(cz_step_opts)]),
        "cz_workspace_size": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _i64p,
                                             ctypes.POINTER(ctypes.c_size_t)]),
        "cz_muon_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, _i64p, _i64p, ctypes.c_float, ctypes.c_float,
                                        ctypes.c_int32, ctypes.c_void_p]),
        "cz_muon_step_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, _i64p, _i64p, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.POINTER(cz_step_opts)]),
        "cz_muon_step_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, _i64p, _i64p, ctypes.c_float, ctypes.c_float,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.POINTER(cz_step_opts)]),
        "cz_device_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, _i32p]),
        "cz_step_programs_built": (ctypes.c_int, [_i64p]),
        "cz_profile_enable": (ctypes.c_int, [ctypes.c_int32]),
        "cz_profile_read": (ctypes.c_int, [_f64p, _i64p, ctypes.c_int32]),
        "cz_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
        "cz_bucket_pack": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _i64p, ctypes.c_int32, ctypes.c_int64,
                                          ctypes.c_void_p, ctypes.c_void_p]),
        "cz_bucket_unpack": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _i64p, ctypes.c_int32, ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_void_p]),
        "cz_apply_update": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, _i64p, _i64p,
                                           ctypes.c_int64, ctypes.c_float, ctypes.c_int32, ctypes.c_void_p]),
        "cz_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "cz_version": (ctypes.c_char_p, []),
        "cz_last_cuda_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _i64(xs: Sequence[int]):
    arr = (ctypes.c_int64 * max(1, len(xs)))(*[int(x) for x in xs])
    return arr


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(fn: str, st: int):
    if st != CZ_OK:
        if st == CZ_ERR_CUDA:
            raise CzError(fn, st, load().cz_last_cuda_error().decode())
        raise CzError(fn, st)


def cz_status_string(status: int) -> str:
    return load().cz_status_string(int(status)).decode()


def cz_version() -> str:
    return load().cz_version().decode()


def cz_last_cuda_error() -> str:
    return load().cz_last_cuda_error().decode()


def cz_make_buckets(numels: Sequence[int], cap_elems: int) -> List[int]:
    lib = load()
    out = (ctypes.c_int64 * max(1, len(numels)))()
    nb = ctypes.c_int64(0)
    _check("cz_make_buckets", lib.cz_make_buckets(_i64(numels), len(numels), int(cap_elems), out, ctypes.byref(nb)))
    return list(out[: nb.value])


class Plan:
    """Owns a cz_plan* (freed with cz_plan_free)."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.cz_plan_free(h)
            self._h = ctypes.c_void_p(0)

    def info(self) -> Tuple[int, int, int]:
        n_p, n_b, R = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        _check("cz_plan_info", load().cz_plan_info(self._h, ctypes.byref(n_p), ctypes.byref(n_b), ctypes.byref(R)))
        return n_p.value, n_b.value, R.value

    def owner(self) -> List[int]:
        n_p, _, _ = self.info()
        out = (ctypes.c_int32 * n_p)()
        _check("cz_plan_owner", load().cz_plan_owner(self._h, out))
        return list(out)

    def cuts(self) -> Tuple[List[List[int]], List[List[int]]]:
        _, n_b, R = self.info()
        pc = (ctypes.c_int64 * (n_b * (R + 1)))()
        ec = (ctypes.c_int64 * (n_b * (R + 1)))()
        _check("cz_plan_cuts", load().cz_plan_cuts(self._h, pc, ec))
        w = R + 1
        return ([list(pc[i * w:(i + 1) * w]) for i in range(n_b)], [list(ec[i * w:(i + 1) * w]) for i in range(n_b)])

    def rank_load(self) -> List[int]:
        _, _, R = self.info()
        out = (ctypes.c_int64 * R)()
        _check("cz_plan_rank_load", load().cz_plan_rank_load(self._h, out))
        return list(out)

    def rank_elems(self) -> List[int]:
        _, _, R = self.info()
        out = (ctypes.c_int64 * R)()
        _check("cz_plan_rank_elems", load().cz_plan_rank_elems(self._h, out))
        return list(out)

    def metrics(self) -> dict:
        r, j, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        _check("cz_plan_metrics", load().cz_plan_metrics(self._h, ctypes.byref(r), ctypes.byref(j), ctypes.byref(c)))
        return {"r_lb": r.value, "j_dp": j.value, "j_comm": c.value}


def cz_plan_partition(numels: Sequence[int], bucket_sizes: Sequence[int], R: int, alpha: float) -> Plan:
    lib = load()
    h = ctypes.c_void_p()
    _check("cz_plan_partition", lib.cz_plan_partition(_i64(numels), len(numels), _i64(bucket_sizes),
                                                      len(bucket_sizes), int(R), float(alpha), ctypes.byref(h)))
    return Plan(h.value)


def cz_plan_partition_cost(numels: Sequence[int], costs: Sequence[int], bucket_sizes: Sequence[int], R: int,
                           alpha: float) -> Plan:
    lib = load()
    h = ctypes.c_void_p()
    _check("cz_plan_partition_cost", lib.cz_plan_partition_cost(_i64(numels), _i64(costs), len(numels),
                                                                _i64(bucket_sizes), len(bucket_sizes), int(R),
                                                                float(alpha), ctypes.byref(h)))
    return Plan(h.value)


def cz_plan_microgroups(costs: Sequence[int], R: int, c_max: int) -> Tuple[List[int], List[int], int]:
    """Returns (group index per tensor, host rank per tensor, number of groups)."""
    n = len(costs)
    g = (ctypes.c_int32 * max(1, n))()
    h = (ctypes.c_int32 * max(1, n))()
    ng = ctypes.c_int64(0)
    _check("cz_plan_microgroups", load().cz_plan_microgroups(_i64(costs), n, int(R), int(c_max), g, h,
                                                             ctypes.byref(ng)))
    return list(g[:n]), list(h[:n]), ng.value


def cz_plan_naive(numels: Sequence[int], bucket_sizes: Sequence[int], R: int) -> Plan:
    lib = load()
    h = ctypes.c_void_p()
    _check("cz_plan_naive", lib.cz_plan_naive(_i64(numels), len(numels), _i64(bucket_sizes), len(bucket_sizes),
                                              int(R), ctypes.byref(h)))
    return Plan(h.value)


def cz_step_opts_default() -> cz_step_opts:
    o = cz_step_opts()
    load().cz_step_opts_default(ctypes.byref(o))
    return o


def _shapes_flat(shapes: Sequence[Tuple[int, int]]):
    flat = []
    for r, c in shapes:
        flat += [int(r), int(c)]
    return _i64(flat)


def cz_workspace_size(plan: Plan, rank: int, shapes: Sequence[Tuple[int, int]]) -> int:
    n = ctypes.c_size_t(0)
    _check("cz_workspace_size", load().cz_workspace_size(plan.handle, int(rank), _shapes_flat(shapes),
                                                         ctypes.byref(n)))
    return n.value


class StepArgs:
    """Host-side marshalled offsets/shapes, reusable across steps."""

    def __init__(self, offsets: Sequence[int], shapes: Sequence[Tuple[int, int]]):
        self.offsets = _i64(offsets)
        self.shapes = _shapes_flat(shapes)
        self.shape_list = [(int(r), int(c)) for r, c in shapes]


def cz_muon_step(plan: Plan, rank: int, flat_param, flat_grad, flat_mom, args: StepArgs, lr: float, mu: float,
                 ns_steps: int, stream=None) -> None:
    st = load().cz_muon_step(plan.handle, int(rank), _ptr(flat_param), _ptr(flat_grad), _ptr(flat_mom),
                             args.offsets, args.shapes, float(lr), float(mu), int(ns_steps), _stream_ptr(stream))
    _check("cz_muon_step", st)


def cz_muon_step_ex(plan: Plan, rank: int, flat_param, flat_grad, flat_mom, args: StepArgs, lr: float, mu: float,
                    ns_steps: int, stream=None, opts: Optional[cz_step_opts] = None) -> None:
    if opts is None:
        opts = cz_step_opts_default()
    st = load().cz_muon_step_ex(plan.handle, int(rank), _ptr(flat_param), _ptr(flat_grad), _ptr(flat_mom),
                                args.offsets, args.shapes, float(lr), float(mu), int(ns_steps), _stream_ptr(stream),
                                ctypes.byref(opts))
    _check("cz_muon_step_ex", st)


CZ_STATIC_WORKSPACE_BYTES = 64 * 1024 * 1024


def cz_muon_step_noalloc(plan: Plan, rank: int, flat_param, flat_grad, flat_mom, args: StepArgs, lr: float,
                         mu: float, ns_steps: int, stream=None, opts: Optional[cz_step_opts] = None) -> None:
    """The step with the library's static device scratch: allocates no device memory."""
    st = load().cz_muon_step_noalloc(plan.handle, int(rank), _ptr(flat_param), _ptr(flat_grad), _ptr(flat_mom),
                                     args.offsets, args.shapes, float(lr), float(mu), int(ns_steps),
                                     _stream_ptr(stream), ctypes.byref(opts) if opts is not None else None)
    _check("cz_muon_step_noalloc", st)


def make_opts(param_bf16=None, workspace=None, workspace_bytes: int = 0, debug_update_out=None,
              grad_is_bf16: bool = False, nesterov: bool = True, eps: Optional[float] = None,
              coeffs: Optional[Tuple[float, float, float]] = None, lr_device=None) -> cz_step_opts:
    """cz_step_opts from the library defaults with the given overrides (tensors are passed by
    data pointer): bf16 parameter copy, caller workspace, debug delta, bf16 gradients, Nesterov,
    eps, Newton-Schulz coefficients (a, b, c), and lr_device, a one-element fp32 device tensor
    read in place of the lr argument (for a learning-rate schedule under a CUDA graph)."""
    o = cz_step_opts_default()
    o.lr_device = _ptr(lr_device)
    o.param_bf16 = _ptr(param_bf16)
    o.workspace = _ptr(workspace)
    o.workspace_bytes = int(workspace_bytes)
    o.debug_update_out = _ptr(debug_update_out)
    o.grad_is_bf16 = 1 if grad_is_bf16 else 0
    o.nesterov = 1 if nesterov else 0
    if eps is not None:
        o.eps = float(eps)
    if coeffs is not None:
        o.a, o.b, o.c = (float(x) for x in coeffs)
    return o


def cz_device_status(stream=None, workspace=None) -> int:
    v = ctypes.c_int32(0)
    _check("cz_device_status", load().cz_device_status(_stream_ptr(stream), _ptr(workspace), ctypes.byref(v)))
    return v.value


def cz_step_programs_built() -> int:
    v = ctypes.c_int64(0)
    _check("cz_step_programs_built", load().cz_step_programs_built(ctypes.byref(v)))
    return v.value


KERNEL_KINDS = ("momentum", "tables", "ns_gram", "ns_poly", "ns_update", "ns_update_apply", "ns_fused",
                "ns_small")


def cz_profile_enable(on: bool) -> None:
    _check("cz_profile_enable", load().cz_profile_enable(1 if on else 0))


def cz_profile_read() -> dict:
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check("cz_profile_read", load().cz_profile_read(ms, cnt, n))
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def cz_selftest_bounded_wait(timeout_ns: int, workspace, stream=None) -> None:
    _check("cz_selftest_bounded_wait", load().cz_selftest_bounded_wait(int(timeout_ns), _ptr(workspace),
                                                                       _stream_ptr(stream)))


def cz_bucket_pack(bucket, elem_cuts: Sequence[int], block: int, padded, stream=None) -> None:
    """Rank r's interval of the bucket -> block r of `padded` (zero tail)."""
    R = len(elem_cuts) - 1
    _check("cz_bucket_pack", load().cz_bucket_pack(_ptr(bucket), int(bucket.element_size()), _i64(elem_cuts), R,
                                                   int(block), _ptr(padded), _stream_ptr(stream)))


def cz_bucket_unpack(padded, elem_cuts: Sequence[int], block: int, bucket, stream=None) -> None:
    """Block r of `padded` (first S_r elements) -> rank r's interval of the bucket."""
    R = len(elem_cuts) - 1
    _check("cz_bucket_unpack", load().cz_bucket_unpack(_ptr(padded), int(padded.element_size()), _i64(elem_cuts), R,
                                                       int(block), _ptr(bucket), _stream_ptr(stream)))


def cz_apply_update(flat_param, param_bf16, flat_update, offsets: Sequence[int], shapes: Sequence[Tuple[int, int]],
                    lr: float, shape_scale: bool = True, stream=None) -> None:
    """W <- W - fp32(lr * sqrt(max(1, rows/cols))) * U per listed tensor (bf16 copy optional)."""
    _check("cz_apply_update", load().cz_apply_update(_ptr(flat_param), _ptr(param_bf16), _ptr(flat_update),
                                                     _i64(offsets), _shapes_flat(shapes), len(offsets), float(lr),
                                                     1 if shape_scale else 0, _stream_ptr(stream)))
