"""Thin ctypes binding of the C ABI in ``include/bmm.h`` (same names).

Argument marshalling only: every step of the product runs in the CUDA
kernels of ``libdmt_bmm.so``.  Device pointers may be passed as integers or
as any object with ``data_ptr()`` (a torch tensor); streams as an integer
handle, an object with ``cuda_stream`` (a torch stream), or None.  There is
no fallback: if the library is not built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

BMM_BF16, BMM_F16, BMM_F32 = 0, 1, 2
DTYPES = {"bf16": BMM_BF16, "f16": BMM_F16, "f32": BMM_F32}

BMM_OK = 0
BMM_ERR_INVALID_ARG = 1
BMM_ERR_UNSUPPORTED = 2
BMM_ERR_MISALIGNED = 3
BMM_ERR_CUDA = 4
BMM_ERR_DEVICE_TIMEOUT = 5
BMM_ERR_NO_DEVICE = 6

EXPORTED = ("bmm_create", "bmm_plan_query", "bmm_get_plan_info", "bmm_run",
            "bmm_get_device_error", "bmm_destroy", "bmm_status_string", "bmm_version",
            "bmm_grouped_create", "bmm_grouped_run", "bmm_grouped_get_device_error",
            "bmm_grouped_get_info", "bmm_grouped_destroy",
            "bmm_attn_create", "bmm_attn_run", "bmm_attn_get_device_error", "bmm_attn_destroy",
            "bmm_host_create", "bmm_host_run", "bmm_host_get_device_error", "bmm_host_get_chunks",
            "bmm_host_destroy")


class bmm_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("batch", "M", "N", "K", "lda", "ldb", "ldc", "strideA", "strideB", "strideC")] + \
               [(n, ctypes.c_int32) for n in ("transA", "transB", "typeA", "typeB", "typeC")]


class bmm_plan_info_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("tile_m", "tile_n", "tile_k", "stages", "swap_ab", "pack_a", "pack_b", "even_k",
                 "tmem_cols", "cta_pair")] + \
               [(n, ctypes.c_int64) for n in
                ("tiles", "smem_bytes", "stage_bytes", "workspace_bytes")] + \
               [("stream_k", ctypes.c_int32), ("sk_tiles", ctypes.c_int32),
                ("sk_workspace_bytes", ctypes.c_int64),
                ("stages_bf16_box", ctypes.c_int32), ("reserved0", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class BmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bmm_status_string(status)} ({status})")


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library() -> ctypes.CDLL:
    """Load ``libdmt_bmm.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"GPU library not built: {path} is missing "
                           "(run dense_matmul_tensor_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    lib.bmm_create.argtypes = [P(bmm_desc_t), P(vp)]
    lib.bmm_create.restype = ctypes.c_int
    lib.bmm_plan_query.argtypes = [P(bmm_desc_t), P(bmm_plan_info_t)]
    lib.bmm_plan_query.restype = ctypes.c_int
    lib.bmm_get_plan_info.argtypes = [vp, P(bmm_plan_info_t)]
    lib.bmm_get_plan_info.restype = ctypes.c_int
    lib.bmm_run.argtypes = [vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp]
    lib.bmm_run.restype = ctypes.c_int
    lib.bmm_get_device_error.argtypes = [vp, P(ctypes.c_uint32)]
    lib.bmm_get_device_error.restype = ctypes.c_int
    lib.bmm_destroy.argtypes = [vp]
    lib.bmm_destroy.restype = ctypes.c_int
    lib.bmm_status_string.argtypes = [ctypes.c_int]
    lib.bmm_status_string.restype = ctypes.c_char_p
    lib.bmm_version.argtypes = []
    lib.bmm_version.restype = ctypes.c_int32
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return ctypes.c_void_p(x.data_ptr())
    return ctypes.c_void_p(int(x))


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return ctypes.c_void_p(s.cuda_stream)
    return ctypes.c_void_p(int(s))


def make_desc(*, batch, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, transA=0, transB=0,
              typeA="bf16", typeB=None, typeC="f32") -> bmm_desc_t:
    t = lambda v: DTYPES[v] if isinstance(v, str) else int(v)  # noqa: E731
    return bmm_desc_t(batch, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, int(transA),
                      int(transB), t(typeA), t(typeB if typeB is not None else typeA), t(typeC))


def bmm_status_string(status: int) -> str:
    return load_library().bmm_status_string(int(status)).decode()


def bmm_version() -> int:
    return load_library().bmm_version()


def bmm_plan_query(desc: bmm_desc_t) -> bmm_plan_info_t:
    info = bmm_plan_info_t()
    st = load_library().bmm_plan_query(ctypes.byref(desc), ctypes.byref(info))
    if st != BMM_OK:
        raise BmmError(st, "bmm_plan_query")
    return info


def bmm_create(desc: bmm_desc_t) -> ctypes.c_void_p:
    plan = ctypes.c_void_p()
    st = load_library().bmm_create(ctypes.byref(desc), ctypes.byref(plan))
    if st != BMM_OK:
        raise BmmError(st, "bmm_create")
    return plan


def bmm_get_plan_info(plan) -> bmm_plan_info_t:
    info = bmm_plan_info_t()
    st = load_library().bmm_get_plan_info(plan, ctypes.byref(info))
    if st != BMM_OK:
        raise BmmError(st, "bmm_get_plan_info")
    return info


def bmm_run(plan, A, B, C, alpha=1.0, beta=0.0, stream=None) -> None:
    st = load_library().bmm_run(plan, _ptr(A), _ptr(B), _ptr(C), float(alpha), float(beta),
                                _stream(stream))
    if st != BMM_OK:
        raise BmmError(st, "bmm_run")


def bmm_get_device_error(plan):
    """Returns (status, raw_word); call after the stream has been synchronised."""
    w = ctypes.c_uint32(0)
    st = load_library().bmm_get_device_error(plan, ctypes.byref(w))
    return st, w.value


def bmm_destroy(plan) -> None:
    st = load_library().bmm_destroy(plan)
    if st != BMM_OK:
        raise BmmError(st, "bmm_destroy")


class Plan:
    """Owns one plan: ``with Plan(desc) as p: p.run(A, B, C, alpha, beta, stream)``."""

    def __init__(self, desc: bmm_desc_t):
        self.desc = desc
        self.handle = bmm_create(desc)

    def run(self, A, B, C, alpha=1.0, beta=0.0, stream=None):
        bmm_run(self.handle, A, B, C, alpha, beta, stream)

    def info(self) -> bmm_plan_info_t:
        return bmm_get_plan_info(self.handle)

    def device_error(self):
        return bmm_get_device_error(self.handle)

    def close(self):
        if self.handle:
            bmm_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bmm_run_noalloc(desc: bmm_desc_t, A, B, C, alpha=1.0, beta=0.0, stream=None,
                    device_error=None) -> None:
    """The allocation-free variant of bmm_run, for callers that cannot call
    cudaMalloc (an allocator owns the device memory, or the call path cannot
    afford cudaMalloc's cost and device synchronisation).  Plans ``desc`` for
    this call and uses only the library's built-in device scratch (32 MiB of
    operand staging plus an error word, shared by all calls: serialise calls
    whose GPU work would overlap); operands that would need more staging are
    read in place by the kernel's row loader.  ``device_error`` is an optional device
    pointer that receives the call's device error word on ``stream``."""
    lib = load_library()
    fn = lib.bmm_run_noalloc
    if fn.argtypes is None:
        vp = ctypes.c_void_p
        fn.argtypes = [ctypes.POINTER(bmm_desc_t), vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp]
        fn.restype = ctypes.c_int
    st = fn(ctypes.byref(desc), _ptr(A), _ptr(B), _ptr(C), float(alpha), float(beta),
            _stream(stream), _ptr(device_error))
    if st != BMM_OK:
        raise BmmError(st, "bmm_run_noalloc")


# ------------------------------------------------------------ grouped launch

class bmm_group_problem_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("M", "N", "K", "lda", "ldb", "ldc")] + \
               [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float)]


def _grouped_lib():
    lib = load_library()
    if lib.bmm_grouped_create.argtypes is None:
        vp, P = ctypes.c_void_p, ctypes.POINTER
        i32 = ctypes.c_int32
        lib.bmm_grouped_create.argtypes = [i32, P(bmm_group_problem_t), i32, i32, i32, i32, P(vp)]
        lib.bmm_grouped_create.restype = ctypes.c_int
        lib.bmm_grouped_run.argtypes = [vp, P(bmm_group_problem_t), vp]
        lib.bmm_grouped_run.restype = ctypes.c_int
        lib.bmm_grouped_get_device_error.argtypes = [vp, P(ctypes.c_uint32)]
        lib.bmm_grouped_get_device_error.restype = ctypes.c_int
        lib.bmm_grouped_get_info.argtypes = [vp, P(i32), P(ctypes.c_int64), P(i32)]
        lib.bmm_grouped_get_info.restype = ctypes.c_int
        lib.bmm_grouped_destroy.argtypes = [vp]
        lib.bmm_grouped_destroy.restype = ctypes.c_int
    return lib


def make_problems(items) -> ctypes.Array:
    """items: iterable of dicts with M, N, K, lda, ldb, ldc, A, B, C, alpha,
    beta (A/B/C as device pointers or tensors)."""
    items = list(items)
    arr = (bmm_group_problem_t * max(len(items), 1))()
    for i, it in enumerate(items):
        arr[i] = bmm_group_problem_t(it["M"], it["N"], it["K"], it["lda"], it["ldb"], it["ldc"],
                                     _ptr(it.get("A")), _ptr(it.get("B")), _ptr(it.get("C")),
                                     float(it.get("alpha", 1.0)), float(it.get("beta", 0.0)))
    return arr, len(items)


def bmm_grouped_create(problems, count, transA=0, transB=0, typeAB="bf16", typeC="f32"):
    plan = ctypes.c_void_p()
    t = lambda v: DTYPES[v] if isinstance(v, str) else int(v)  # noqa: E731
    st = _grouped_lib().bmm_grouped_create(int(count), problems, int(transA), int(transB), t(typeAB),
                                           t(typeC), ctypes.byref(plan))
    if st != BMM_OK:
        raise BmmError(st, "bmm_grouped_create")
    return plan


def bmm_grouped_run(plan, problems, stream=None):
    st = _grouped_lib().bmm_grouped_run(plan, problems, _stream(stream))
    if st != BMM_OK:
        raise BmmError(st, "bmm_grouped_run")


def bmm_grouped_get_device_error(plan):
    w = ctypes.c_uint32(0)
    st = _grouped_lib().bmm_grouped_get_device_error(plan, ctypes.byref(w))
    return st, w.value


def bmm_grouped_get_info(plan):
    tn, tiles, stages = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
    st = _grouped_lib().bmm_grouped_get_info(plan, ctypes.byref(tn), ctypes.byref(tiles),
                                             ctypes.byref(stages))
    if st != BMM_OK:
        raise BmmError(st, "bmm_grouped_get_info")
    return {"tile_n": tn.value, "tiles": tiles.value, "stages": stages.value}


def bmm_grouped_destroy(plan):
    st = _grouped_lib().bmm_grouped_destroy(plan)
    if st != BMM_OK:
        raise BmmError(st, "bmm_grouped_destroy")


# ------------------------------------------------------------ fused attention

class bmm_attn_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("batch", "Lq", "Lk", "D", "ldq", "ldk", "ldv", "ldo",
                                              "strideQ", "strideK", "strideV", "strideO")] + \
               [("alpha", ctypes.c_float)]


def make_attn_desc(*, batch, Lq, Lk, D=128, alpha, ldq=None, ldk=None, ldv=None, ldo=None,
                   strideQ=None, strideK=None, strideV=None, strideO=None) -> bmm_attn_desc_t:
    """Descriptor of O = softmax(alpha Q K^T) V; dense strides by default."""
    ldq, ldk, ldv, ldo = (x if x is not None else D for x in (ldq, ldk, ldv, ldo))
    sq = strideQ if strideQ is not None else Lq * ldq
    sk = strideK if strideK is not None else Lk * ldk
    sv = strideV if strideV is not None else Lk * ldv
    so = strideO if strideO is not None else Lq * ldo
    return bmm_attn_desc_t(batch, Lq, Lk, D, ldq, ldk, ldv, ldo, sq, sk, sv, so, float(alpha))


def _attn_lib():
    lib = load_library()
    if lib.bmm_attn_create.argtypes is None:
        vp, P = ctypes.c_void_p, ctypes.POINTER
        lib.bmm_attn_create.argtypes = [P(bmm_attn_desc_t), P(vp)]
        lib.bmm_attn_create.restype = ctypes.c_int
        lib.bmm_attn_run.argtypes = [vp, vp, vp, vp, vp, vp]
        lib.bmm_attn_run.restype = ctypes.c_int
        lib.bmm_attn_get_device_error.argtypes = [vp, P(ctypes.c_uint32)]
        lib.bmm_attn_get_device_error.restype = ctypes.c_int
        lib.bmm_attn_destroy.argtypes = [vp]
        lib.bmm_attn_destroy.restype = ctypes.c_int
    return lib


def bmm_attn_create(desc: bmm_attn_desc_t):
    plan = ctypes.c_void_p()
    st = _attn_lib().bmm_attn_create(ctypes.byref(desc), ctypes.byref(plan))
    if st != BMM_OK:
        raise BmmError(st, "bmm_attn_create")
    return plan


def bmm_attn_run(plan, Q, K, V, O, stream=None):
    st = _attn_lib().bmm_attn_run(plan, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _stream(stream))
    if st != BMM_OK:
        raise BmmError(st, "bmm_attn_run")


def bmm_attn_get_device_error(plan):
    w = ctypes.c_uint32(0)
    st = _attn_lib().bmm_attn_get_device_error(plan, ctypes.byref(w))
    return st, w.value


def bmm_attn_destroy(plan):
    st = _attn_lib().bmm_attn_destroy(plan)
    if st != BMM_OK:
        raise BmmError(st, "bmm_attn_destroy")


class AttnPlan:
    """Owns one attention plan: ``with AttnPlan(desc) as p: p.run(Q, K, V, O, stream)``."""

    def __init__(self, desc: bmm_attn_desc_t):
        self.desc = desc
        self.handle = bmm_attn_create(desc)

    def run(self, Q, K, V, O, stream=None):
        bmm_attn_run(self.handle, Q, K, V, O, stream)

    def device_error(self):
        return bmm_attn_get_device_error(self.handle)

    def close(self):
        if self.handle:
            bmm_attn_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------ host buffers

def _host_lib():
    lib = load_library()
    if lib.bmm_host_create.argtypes is None:
        vp, P, i32 = ctypes.c_void_p, ctypes.POINTER, ctypes.c_int32
        lib.bmm_host_create.argtypes = [P(bmm_desc_t), i32, P(vp)]
        lib.bmm_host_create.restype = ctypes.c_int
        lib.bmm_host_run.argtypes = [vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp]
        lib.bmm_host_run.restype = ctypes.c_int
        lib.bmm_host_get_device_error.argtypes = [vp, P(ctypes.c_uint32)]
        lib.bmm_host_get_device_error.restype = ctypes.c_int
        lib.bmm_host_get_chunks.argtypes = [vp, P(i32), P(i32)]
        lib.bmm_host_get_chunks.restype = ctypes.c_int
        lib.bmm_host_destroy.argtypes = [vp]
        lib.bmm_host_destroy.restype = ctypes.c_int
    return lib


class HostPlan:
    """C = alpha op(A) op(B) + beta C from and to host memory, transfers
    overlapped with the computation: ``with HostPlan(desc) as p: p.run(hA,
    hB, hC, alpha, beta, stream)`` (hA, hB, hC: CPU tensors, ideally pinned)."""

    def __init__(self, desc: bmm_desc_t, chunks: int = 0):
        self.desc = desc
        self.handle = ctypes.c_void_p()
        st = _host_lib().bmm_host_create(ctypes.byref(desc), int(chunks), ctypes.byref(self.handle))
        if st != BMM_OK:
            self.handle = None
            raise BmmError(st, "bmm_host_create")

    def run(self, A, B, C, alpha=1.0, beta=0.0, stream=None):
        st = _host_lib().bmm_host_run(self.handle, _ptr(A), _ptr(B), _ptr(C), float(alpha),
                                      float(beta), _stream(stream))
        if st != BMM_OK:
            raise BmmError(st, "bmm_host_run")

    def chunks(self):
        c, r = ctypes.c_int32(), ctypes.c_int32()
        _host_lib().bmm_host_get_chunks(self.handle, ctypes.byref(c), ctypes.byref(r))
        return c.value, bool(r.value)

    def device_error(self):
        w = ctypes.c_uint32(0)
        st = _host_lib().bmm_host_get_device_error(self.handle, ctypes.byref(w))
        return st, w.value

    def close(self):
        if self.handle:
            _host_lib().bmm_host_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
