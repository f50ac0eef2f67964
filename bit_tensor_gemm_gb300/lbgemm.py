"""Python binding of the C ABI in ``include/lbgemm.h`` (argument marshalling only).

Every function has the name of its C entry point.  Pointer arguments accept a
plain integer address or any object with ``data_ptr()`` (a torch tensor);
``stream`` accepts an integer handle, an object with ``cuda_stream`` (a
torch.cuda.Stream), or None for torch's current stream when torch is loaded
(else the legacy default stream).  A non-OK status raises ``LbgemmError``
with the library's message.  There is no fallback: if the compiled library
is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "lib", "liblbgemm.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_ALIGNMENT = 2
ERR_UNSUPPORTED = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_WORKSPACE = 6

# kernels of the default dispatch (lbgemm_route)
ROUTE_TABLE, ROUTE_POPC, ROUTE_SKINNY, ROUTE_WARPMMA, ROUTE_SMALL, ROUTE_FUSED, ROUTE_NONE = range(7)
ROUTE_STREAM = 7
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "ALIGNMENT", 3: "UNSUPPORTED", 4: "CUDA",
                5: "TIMEOUT", 6: "WORKSPACE"}


class LbgemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"lbgemm {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_i64, _i32, _vp, _f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
_SIGNATURES = {
    "lbgemm_num_variants": (_i32, []),
    "lbgemm_default_variant": (_i32, []),
    "lbgemm_variant_info": (_i32, [_i32, _i32, _vp, _vp, _vp, _vp]),
    "lbgemm_run": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "lbgemm_run_variant": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "lbgemm_run_fused": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "lbgemm_run_warpmma": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "lbgemm_run_tile": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _i32, _vp]),
    "lbgemm_workspace_size": (ctypes.c_size_t, [_i32, _i64, _i64, _i64]),
    "lbgemm_run_ws": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp, ctypes.c_size_t,
                             _vp]),
    "lbgemm_run_popc": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "lbgemm_run_static": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "lbgemm_encoded_size": (ctypes.c_size_t, [_i32, _i64, _i64]),
    "lbgemm_encode": (_i32, [_i32, _i64, _i64, _vp, _vp, _vp]),
    "lbgemm_run_encoded": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "lbgemm_linear": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "lbgemm_quantize_rows": (_i32, [_i64, _i64, _vp, _vp, _vp, _vp]),
    "lbgemm_linear_quant": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "lbgemm_linear_variant": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _i32, _vp]),
    "lbgemm_linear_candidate": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                       _vp]),
    "lbgemm_select": (_i32, [_i32, _i64, _i64, _i64]),
    "lbgemm_table_set": (_i32, [_i32, _i64, _i64, _i64, _i32]),
    "lbgemm_select_for": (_i32, [_i32, _i32, _i64, _i64, _i64]),
    "lbgemm_route": (_i32, [_i32, _i64, _i64, _i64, _i32, _vp]),
    "lbgemm_dispatch_for": (_i32, [_i32, _i32, _i64, _i64, _i64, _vp]),
    "lbgemm_candidates": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _i32]),
    "lbgemm_run_candidate": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _i32, _vp]),
    "lbgemm_time_candidates": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp, _vp, _i32,
                                      _i32, _i32, _vp, _vp]),
    "lbgemm_table_set_choice_for": (_i32, [_i32, _i32, _i64, _i64, _i64, _i32, _i32, _i32]),
    "lbgemm_table_get_for": (_i32, [_i32, _i32, _i64, _i64, _i64, _vp, _vp, _vp]),
    "lbgemm_table_default_path": (ctypes.c_char_p, []),
    "lbgemm_table_set_for": (_i32, [_i32, _i32, _i64, _i64, _i64, _i32]),
    "lbgemm_table_clear": (_i32, []),
    "lbgemm_table_size": (_i64, []),
    "lbgemm_table_load": (_i32, [ctypes.c_char_p]),
    "lbgemm_table_save": (_i32, [ctypes.c_char_p]),
    "lbgemm_choose": (_i32, [_vp, _i32, _f32]),
    "lbgemm_choose_candidate": (_i32, [_vp, _i32, _i32, _f32]),
    "lbgemm_mlp_load": (_i32, [ctypes.c_char_p]),
    "lbgemm_mlp_clear": (_i32, []),
    "lbgemm_mlp_predict": (_i32, [_i32, _i64, _i64, _i64, _i32, _vp]),
    "lbgemm_time_variants": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _vp,
                                    _vp]),
    "lbgemm_run_host": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "lbgemm_set_exact_chunk": (_i32, [_i32, _i32]),
    "lbgemm_get_exact_chunk": (_i32, [_i32]),
    "lbgemm_set_tail_split": (_i32, [_i32]),
    "lbgemm_set_fused_slice": (_i32, [_i32]),
    "lbgemm_get_fused_slice": (_i32, []),
    "lbgemm_set_fused_stream_k": (_i32, [_i32]),
    "lbgemm_fused_schedule": (_i32, [_i64, _i64, _i64, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_int),
                                     ctypes.POINTER(ctypes.c_int)]),
    "lbgemm_get_fused_stream_k": (_i32, []),
    "lbgemm_get_tail_split": (_i32, []),
    "lbgemm_device_status": (_i32, [_vp]),
    "lbgemm_selftest_timeout": (_i32, [_vp]),
    "lbgemm_last_error": (ctypes.c_char_p, []),
    "lbgemm_launch_count": (_i64, []),
}

_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Open the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIBRARY
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; "
                    "g.build()' or python bit_tensor_gemm_gb300/build.py)")
            lib = ctypes.CDLL(p)
            for name, (res, args) in _SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            if path is not None:
                return lib
            _lib = lib
    return _lib


def exported_symbols():
    return sorted(_SIGNATURES)


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):  # numpy array (host memory)
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch  # noqa: PLC0415
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError(f"not a stream: {type(s).__name__}")


def _check(status: int) -> None:
    if status != OK:
        raise LbgemmError(status, (load().lbgemm_last_error() or b"").decode())


# ---- entry points -------------------------------------------------------------

def lbgemm_num_variants() -> int:
    return load().lbgemm_num_variants()


def lbgemm_default_variant() -> int:
    return load().lbgemm_default_variant()


def lbgemm_variant_info(bits: int, variant: int) -> dict:
    vals = [ctypes.c_int() for _ in range(4)]
    _check(load().lbgemm_variant_info(bits, variant, *[ctypes.addressof(v) for v in vals]))
    return dict(zip(("tile_m", "tile_n", "tile_k", "stages"), (v.value for v in vals)))


def lbgemm_run(bits, M, N, K, A, B, C, stream=None) -> None:
    _check(load().lbgemm_run(bits, M, N, K, _addr(A), _addr(B), _addr(C), _stream(stream)))


def lbgemm_run_variant(bits, M, N, K, A, B, C, variant, stream=None) -> None:
    _check(load().lbgemm_run_variant(bits, M, N, K, _addr(A), _addr(B), _addr(C), variant,
                                     _stream(stream)))


def lbgemm_run_fused(M, N, K, A, B, C, tile_n=128, stream=None) -> None:
    _check(load().lbgemm_run_fused(M, N, K, _addr(A), _addr(B), _addr(C), tile_n, _stream(stream)))


def lbgemm_run_warpmma(M, N, K, A, B, C, stream=None) -> None:
    _check(load().lbgemm_run_warpmma(M, N, K, _addr(A), _addr(B), _addr(C), _stream(stream)))


def lbgemm_run_tile(bits, M, N, K, A, B, C, tile, stages, stream=None) -> None:
    _check(load().lbgemm_run_tile(bits, M, N, K, _addr(A), _addr(B), _addr(C), tile, stages,
                                  _stream(stream)))


def lbgemm_workspace_size(bits, M, N, K) -> int:
    return load().lbgemm_workspace_size(bits, M, N, K)


def lbgemm_run_ws(bits, M, N, K, A, B, C, variant, workspace, workspace_bytes, stream=None):
    _check(load().lbgemm_run_ws(bits, M, N, K, _addr(A), _addr(B), _addr(C), variant,
                                _addr(workspace), workspace_bytes, _stream(stream)))


def lbgemm_run_popc(M, N, K, A, B, C, variant=-1, stream=None) -> None:
    _check(load().lbgemm_run_popc(M, N, K, _addr(A), _addr(B), _addr(C), variant,
                                  _stream(stream)))


STATIC_SCRATCH_BYTES = 32 << 20  # LBGEMM_STATIC_SCRATCH_BYTES in lbgemm.h


def lbgemm_run_static(bits, M, N, K, A, B, C, variant=-1, stream=None) -> None:
    """lbgemm_run_variant with the library's fixed scratch array: allocates nothing."""
    _check(load().lbgemm_run_static(bits, M, N, K, _addr(A), _addr(B), _addr(C), variant,
                                    _stream(stream)))


def lbgemm_encoded_size(bits, rows, K) -> int:
    return load().lbgemm_encoded_size(bits, rows, K)


def lbgemm_encode(bits, rows, K, src, dst, stream=None) -> None:
    _check(load().lbgemm_encode(bits, rows, K, _addr(src), _addr(dst), _stream(stream)))


def lbgemm_run_encoded(bits, M, N, K, A_enc, B_enc, C, variant=-1, stream=None) -> None:
    _check(load().lbgemm_run_encoded(bits, M, N, K, _addr(A_enc), _addr(B_enc), _addr(C), variant,
                                     _stream(stream)))


def lbgemm_linear(M, N, K, X, sx, W, sw, Y, stream=None) -> None:
    _check(load().lbgemm_linear(M, N, K, _addr(X), _addr(sx), _addr(W), _addr(sw), _addr(Y),
                                _stream(stream)))


def lbgemm_quantize_rows(M, K, X, Q, S, stream=None) -> None:
    _check(load().lbgemm_quantize_rows(M, K, _addr(X), _addr(Q), _addr(S), _stream(stream)))


def lbgemm_linear_quant(M, N, K, X, W, sw, Y, stream=None) -> None:
    _check(load().lbgemm_linear_quant(M, N, K, _addr(X), _addr(W), _addr(sw), _addr(Y),
                                      _stream(stream)))


def lbgemm_linear_variant(M, N, K, X, sx, W, sw, Y, variant, stream=None) -> None:
    _check(load().lbgemm_linear_variant(M, N, K, _addr(X), _addr(sx), _addr(W), _addr(sw),
                                        _addr(Y), variant, _stream(stream)))


def lbgemm_linear_candidate(M, N, K, X, sx, W, sw, Y, route, param=0, stream=None) -> None:
    _check(load().lbgemm_linear_candidate(M, N, K, _addr(X), _addr(sx), _addr(W), _addr(sw),
                                          _addr(Y), route, param, _stream(stream)))


def lbgemm_select(bits, M, N, K) -> int:
    return load().lbgemm_select(bits, M, N, K)


def lbgemm_select_for(sm_count, bits, M, N, K) -> int:
    return load().lbgemm_select_for(sm_count, bits, M, N, K)


def lbgemm_route(bits, M, N, K, linear=False):
    """(route, tile_n) of the default dispatch for 16-byte-aligned operands."""
    t = ctypes.c_int(0)
    r = load().lbgemm_route(bits, M, N, K, int(bool(linear)), ctypes.byref(t))
    if r < 0:
        raise LbgemmError(ERR_INVALID_ARG, f"lbgemm_route({bits}, {M}, {N}, {K}): bad arguments")
    return r, t.value


def lbgemm_dispatch_for(sm_count, bits, M, N, K):
    """(route, param) that lbgemm_run runs for 16-byte-aligned operands on a
    device with sm_count SMs: the table's measured route, else the shape rules."""
    prm = ctypes.c_int(0)
    r = load().lbgemm_dispatch_for(sm_count, bits, M, N, K, ctypes.byref(prm))
    if r < 0:
        raise LbgemmError(ERR_INVALID_ARG, f"lbgemm_dispatch_for({bits}, {M}, {N}, {K}): bad arguments")
    return r, prm.value


def lbgemm_candidates(bits, M, N, K) -> list:
    """The (route, param) candidates the timing sweep measures for a shape."""
    n = load().lbgemm_candidates(bits, M, N, K, None, None, 0)
    if n < 0:
        raise LbgemmError(ERR_INVALID_ARG, f"lbgemm_candidates({bits}, {M}, {N}, {K}): bad arguments")
    routes, params = (ctypes.c_int * n)(), (ctypes.c_int * n)()
    load().lbgemm_candidates(bits, M, N, K, ctypes.addressof(routes), ctypes.addressof(params), n)
    return list(zip(routes, params))


def lbgemm_run_candidate(bits, M, N, K, A, B, C, route, param, stream=None) -> None:
    _check(load().lbgemm_run_candidate(bits, M, N, K, _addr(A), _addr(B), _addr(C), route, param,
                                       _stream(stream)))


def lbgemm_time_candidates(bits, M, N, K, A, B, C, candidates, warmup=1, reps=5, flush_l2=True,
                           stream=None) -> list:
    """Median milliseconds of each (route, param) candidate, interleaved runs."""
    n = len(candidates)
    routes = (ctypes.c_int * n)(*[int(r) for r, _ in candidates])
    params = (ctypes.c_int * n)(*[int(p) for _, p in candidates])
    times = (ctypes.c_float * n)()
    _check(load().lbgemm_time_candidates(bits, M, N, K, _addr(A), _addr(B), _addr(C), n,
                                         ctypes.addressof(routes), ctypes.addressof(params),
                                         warmup, reps, int(bool(flush_l2)),
                                         ctypes.addressof(times), _stream(stream)))
    return list(times)


def lbgemm_table_set_choice_for(sm_count, bits, M, N, K, variant, route=-1, param=0) -> None:
    _check(load().lbgemm_table_set_choice_for(sm_count, bits, M, N, K, variant, route, param))


def lbgemm_table_get_for(sm_count, bits, M, N, K):
    """(variant, route, param) of the exact entry (route -1: none), or None."""
    v, r, p = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    got = load().lbgemm_table_get_for(sm_count, bits, M, N, K, ctypes.byref(v), ctypes.byref(r),
                                      ctypes.byref(p))
    if got < 0:
        raise LbgemmError(ERR_INVALID_ARG, "lbgemm_table_get_for: bad arguments")
    return (v.value, r.value, p.value) if got else None


def lbgemm_table_default_path() -> str:
    return (load().lbgemm_table_default_path() or b"").decode()


def lbgemm_table_set(bits, M, N, K, variant) -> None:
    _check(load().lbgemm_table_set(bits, M, N, K, variant))


def lbgemm_table_set_for(sm_count, bits, M, N, K, variant) -> None:
    _check(load().lbgemm_table_set_for(sm_count, bits, M, N, K, variant))


def lbgemm_table_clear() -> None:
    _check(load().lbgemm_table_clear())


def lbgemm_table_size() -> int:
    return load().lbgemm_table_size()


def lbgemm_table_load(path: str) -> None:
    _check(load().lbgemm_table_load(os.fsencode(path)))


def lbgemm_table_save(path: str) -> None:
    _check(load().lbgemm_table_save(os.fsencode(path)))


def lbgemm_mlp_load(path: str) -> None:
    _check(load().lbgemm_mlp_load(os.fsencode(path)))


def lbgemm_mlp_clear() -> None:
    _check(load().lbgemm_mlp_clear())


def lbgemm_mlp_predict(bits, M, N, K, sm_count) -> tuple[int, int]:
    """(top class, second class) of the loaded network, (-1, -1) if none."""
    second = ctypes.c_int(-1)
    first = load().lbgemm_mlp_predict(bits, M, N, K, sm_count, ctypes.addressof(second))
    return first, (second.value if first >= 0 else -1)


def lbgemm_choose(times, default_variant: int = 7, keep_within: float = 0.02) -> int:
    arr = (ctypes.c_float * 9)(*[float(t) for t in times])
    return load().lbgemm_choose(ctypes.addressof(arr), default_variant, keep_within)


def lbgemm_choose_candidate(times, default_index: int = 7, keep_within: float = 0.02) -> int:
    arr = (ctypes.c_float * len(times))(*[float(t) for t in times])
    return load().lbgemm_choose_candidate(ctypes.addressof(arr), len(times), default_index,
                                          keep_within)


def lbgemm_time_variants(bits, M, N, K, A, B, C, warmup=2, reps=5, flush_l2=True,
                         stream=None) -> list:
    arr = (ctypes.c_float * 9)()
    _check(load().lbgemm_time_variants(bits, M, N, K, _addr(A), _addr(B), _addr(C), warmup, reps,
                                       int(bool(flush_l2)), ctypes.addressof(arr),
                                       _stream(stream)))
    return list(arr)


def lbgemm_run_host(bits, M, N, K, A_host, B_host, C_host, variant=-1, stream=None) -> None:
    _check(load().lbgemm_run_host(bits, M, N, K, _addr(A_host), _addr(B_host), _addr(C_host),
                                  variant, _stream(stream)))


def lbgemm_set_exact_chunk(bits: int, k_elems: int) -> None:
    _check(load().lbgemm_set_exact_chunk(bits, k_elems))


def lbgemm_get_exact_chunk(bits: int) -> int:
    return load().lbgemm_get_exact_chunk(bits)


def lbgemm_set_tail_split(mode: int) -> None:
    """0 whole-problem splits only, 1 also a partial last wave (default), 2 forced."""
    _check(load().lbgemm_set_tail_split(mode))


def lbgemm_set_fused_slice(k_elems: int) -> None:
    """K elements per slice of the 64/128-wide in-kernel-conversion kernels
    (128 or 256; 0 = by tile width, the default)."""
    _check(load().lbgemm_set_fused_slice(k_elems))


def lbgemm_get_fused_slice() -> int:
    return load().lbgemm_get_fused_slice()


def lbgemm_set_fused_stream_k(mode: int) -> None:
    """Work schedule of the 64/128-wide in-kernel-conversion kernels: 0 split
    K by the cost model (default), 1 stream-K where possible."""
    _check(load().lbgemm_set_fused_stream_k(mode))


def lbgemm_get_fused_stream_k() -> int:
    return load().lbgemm_get_fused_stream_k()


def lbgemm_fused_schedule(M, N, K, tile_n, linear=False, sm_count=152):
    """(splits, stream_pieces) of the 64/128-wide in-kernel-conversion kernel
    for this GEMM or linear layer on sm_count SMs (host only)."""
    sp, pc = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().lbgemm_fused_schedule(M, N, K, tile_n, int(bool(linear)), sm_count,
                                        ctypes.byref(sp), ctypes.byref(pc)))
    return sp.value, pc.value


def lbgemm_get_tail_split() -> int:
    return load().lbgemm_get_tail_split()


def lbgemm_device_status(stream=None) -> None:
    _check(load().lbgemm_device_status(_stream(stream)))


def lbgemm_selftest_timeout(stream=None) -> None:
    _check(load().lbgemm_selftest_timeout(_stream(stream)))


def lbgemm_last_error() -> str:
    return (load().lbgemm_last_error() or b"").decode()


def lbgemm_launch_count() -> int:
    return load().lbgemm_launch_count()
