"""Python binding of libspecverify: the speculative-decoding verify step on GB300.

A thin ctypes layer over the C ABI in include/specverify.h: every function here
only marshals arguments (device pointers, sizes, the current CUDA stream) and
calls the C entry point of the same name; all arithmetic runs in the library's
CUDA kernels.  Tensor arguments may be torch CUDA tensors (their data pointer
is used) or raw integer device addresses.  Failures raise SpecError with the
library's message.  If the shared library has not been built, loading it
raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "SpecError", "Context", "lib", "spec_create", "spec_destroy", "spec_sync_status",
    "qgemm_w4a16", "qgemm_w8a16", "fwht_rotate", "spec_softmax", "spec_accept",
    "spec_accept_noalloc", "spec_accept_tree", "spec_gumbel_sample", "spec_accept_gumbel",
    "qdequant_w4", "qdequant_w8", "SYMBOLS", "LIB_PATH",
    "SPEC_DTYPE_BF16", "SPEC_DTYPE_F32", "SPEC_QUANT_W4", "SPEC_QUANT_W8",
    "GemmDesc", "GemmStack", "qgemm_stack_create", "qgemm_stack_run", "qgemm_stack_destroy",
    "spec_set_stream_prefetch", "spec_test_stall", "spec_set_gemm_engine",
    "SPEC_GEMM_ENGINE_AUTO", "SPEC_GEMM_ENGINE_SPLIT", "SPEC_GEMM_ENGINE_STACK",
    "spec_repack_w4_codes",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspecverify.so")

SPEC_DTYPE_BF16 = 0
SPEC_DTYPE_F32 = 1
SPEC_QUANT_W4 = 0
SPEC_QUANT_W8 = 1
SPEC_GEMM_ENGINE_AUTO = 0
SPEC_GEMM_ENGINE_SPLIT = 1
SPEC_GEMM_ENGINE_STACK = 2

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64


class GemmDesc(ctypes.Structure):
    """spec_gemm_desc: one GEMM of a stack (field order as in the header)."""
    _fields_ = [("quant", _I), ("qcodes", _P), ("scales", _P), ("zeros", _P), ("group_size", _I),
                ("x", _P), ("y", _P), ("y_dtype", _I), ("T", _I), ("N", _I), ("K", _I),
                ("signs", _P), ("hadamard_block", _I), ("wait_prev", _I)]

# name -> argtypes (all return int status, except spec_last_error / spec_version)
_SIGS = {
    "spec_version": [],
    "spec_last_error": [],
    "spec_create": [_I, _SZ, ctypes.POINTER(_P)],
    "spec_destroy": [_P],
    "spec_sync_status": [_P, _P],
    "qgemm_w4a16": [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _I, _P],
    "qgemm_w8a16": [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _I, _P],
    "fwht_rotate": [_P, _P, _P, _I, _I, _P, _I, _P],
    "spec_softmax": [_P, _P, _P, _I, _I, _P],
    "spec_accept": [_P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P],
    "spec_accept_noalloc": [_P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P],
    "spec_accept_tree": [_P, _P, _P, _P, _I, _I, _P, _P, _P, _P],
    "spec_gumbel_sample": [_P, _P, _I, _I, _U64, _U64, _P, _P, _P],
    "spec_accept_gumbel": [_P, _P, _P, _I, _I, _U64, _U64, _P, _P, _P, _P],
    "qgemm_stack_create": [_P, ctypes.POINTER(GemmDesc), _I, ctypes.POINTER(_P)],
    "qgemm_stack_run": [_P, _P, _P],
    "qgemm_stack_destroy": [_P],
    "spec_set_stream_prefetch": [_P, _I, _I],
    "spec_test_stall": [_P, _I, _U64],
    "spec_set_gemm_engine": [_P, _I],
    "qdequant_w4": [_P, _P, _P, _P, _I, _I, _I, _P, _P],
    "qdequant_w8": [_P, _P, _P, _I, _I, _I, _P, _P],
    "spec_repack_w4_codes": [_P, _P, _I, _I],
}
SYMBOLS = tuple(_SIGS)

_lib = None


class SpecError(RuntimeError):
    def __init__(self, name: str, status: int, message: str):
        super().__init__(f"{name} failed with status {status}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libspecverify.so (built in-tree by build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with bit_qgemm_w4_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name == "spec_last_error" else ctypes.c_int
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name: str, *args) -> None:
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise SpecError(name, rc, lib().spec_last_error().decode())


class Context:
    """Owns a spec_ctx (device workspace + error word) for one stream user."""

    def __init__(self, device: int = 0, workspace_bytes: int = 0):
        h = _P()
        _call("spec_create", device, workspace_bytes, ctypes.byref(h))
        self.handle = h.value
        self.device = device

    def close(self) -> None:
        if self.handle:
            _call("spec_destroy", self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def _h(ctx) -> int:
    return ctx.handle if isinstance(ctx, Context) else int(ctx)


def spec_create(device: int = 0, workspace_bytes: int = 0) -> Context:
    return Context(device, workspace_bytes)


def spec_destroy(ctx: Context) -> None:
    ctx.close()


def spec_sync_status(ctx, stream=None) -> None:
    _call("spec_sync_status", _h(ctx), _stream(stream))


def qgemm_w4a16(ctx, qcodes, scales, zeros, group_size, x, y, T, N, K, signs=None,
                hadamard_block=0, stream=None, y_f32=None) -> None:
    if y_f32 is None:
        y_f32 = str(getattr(y, "dtype", "")) == "torch.float32"
    _call("qgemm_w4a16", _h(ctx), _ptr(qcodes), _ptr(scales), _ptr(zeros), group_size, _ptr(x),
          _ptr(y), SPEC_DTYPE_F32 if y_f32 else SPEC_DTYPE_BF16, T, N, K, _ptr(signs),
          hadamard_block, _stream(stream))


def qgemm_w8a16(ctx, qcodes, scales, group_size, x, y, T, N, K, signs=None, hadamard_block=0,
                stream=None, y_f32=None) -> None:
    if y_f32 is None:
        y_f32 = str(getattr(y, "dtype", "")) == "torch.float32"
    _call("qgemm_w8a16", _h(ctx), _ptr(qcodes), _ptr(scales), group_size, _ptr(x), _ptr(y),
          SPEC_DTYPE_F32 if y_f32 else SPEC_DTYPE_BF16, T, N, K, _ptr(signs), hadamard_block,
          _stream(stream))


def _desc(d: dict) -> GemmDesc:
    y = d["y"]
    y_f32 = d.get("y_f32")
    if y_f32 is None:
        y_f32 = str(getattr(y, "dtype", "")) == "torch.float32"
    return GemmDesc(d.get("quant", SPEC_QUANT_W4), _ptr(d["qcodes"]), _ptr(d["scales"]),
                    _ptr(d.get("zeros")), d["group_size"], _ptr(d["x"]), _ptr(y),
                    SPEC_DTYPE_F32 if y_f32 else SPEC_DTYPE_BF16, d["T"], d["N"], d["K"],
                    _ptr(d.get("signs")), d.get("hadamard_block", 0), d.get("wait_prev", 1))


class GemmStack:
    """Owns a spec_gemm_stack: a list of GEMMs run by one launch."""

    def __init__(self, ctx, descs):
        arr = (GemmDesc * len(descs))(*[_desc(d) for d in descs])
        h = _P()
        _call("qgemm_stack_create", _h(ctx), arr, len(descs), ctypes.byref(h))
        self.handle = h.value
        self.ctx = ctx
        self.n = len(descs)

    def run(self, stream=None) -> None:
        _call("qgemm_stack_run", _h(self.ctx), self.handle, _stream(stream))

    def close(self) -> None:
        if self.handle:
            _call("qgemm_stack_destroy", self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def qgemm_stack_create(ctx, descs) -> GemmStack:
    """descs: dicts with the keys of spec_gemm_desc (quant, qcodes, scales, zeros,
    group_size, x, y, T, N, K, optional signs, hadamard_block, wait_prev (default 1),
    y_f32 (default: from y's dtype))."""
    return GemmStack(ctx, descs)


def qgemm_stack_run(ctx, stack: GemmStack, stream=None) -> None:
    _call("qgemm_stack_run", _h(ctx), stack.handle, _stream(stream))


def qgemm_stack_destroy(stack: GemmStack) -> None:
    stack.close()


def spec_set_stream_prefetch(ctx, lead: int, lead_when_full: int) -> None:
    _call("spec_set_stream_prefetch", _h(ctx), lead, lead_when_full)


def spec_test_stall(ctx, skip_unit: int, wait_limit_ns: int) -> None:
    _call("spec_test_stall", _h(ctx), skip_unit, wait_limit_ns)


def spec_set_gemm_engine(ctx, engine: int) -> None:
    _call("spec_set_gemm_engine", _h(ctx), engine)


def fwht_rotate(ctx, x, y, T, K, signs, block, stream=None) -> None:
    _call("fwht_rotate", _h(ctx), _ptr(x), _ptr(y), T, K, _ptr(signs), block, _stream(stream))


def spec_softmax(ctx, logits, probs, rows, V, stream=None) -> None:
    _call("spec_softmax", _h(ctx), _ptr(logits), _ptr(probs), rows, V, _stream(stream))


def spec_accept(ctx, target_logits, draft_probs, draft_tokens, uniforms, T, V, n_accepted,
                out_tokens, near_tie_flags=None, stream=None) -> None:
    _call("spec_accept", _h(ctx), _ptr(target_logits), _ptr(draft_probs), _ptr(draft_tokens),
          _ptr(uniforms), T, V, _ptr(n_accepted), _ptr(out_tokens), _ptr(near_tie_flags),
          _stream(stream))


def spec_accept_noalloc(target_logits, draft_probs, draft_tokens, uniforms, T, V, n_accepted,
                        out_tokens, near_tie_flags=None, device_status=None, stream=None) -> None:
    """spec_accept on the current device with no context and no device allocation
    (T <= 64; see the header for who needs it and how concurrent calls race)."""
    _call("spec_accept_noalloc", _ptr(target_logits), _ptr(draft_probs), _ptr(draft_tokens),
          _ptr(uniforms), T, V, _ptr(n_accepted), _ptr(out_tokens), _ptr(near_tie_flags),
          _ptr(device_status), _stream(stream))


def spec_accept_tree(ctx, target_logits, draft_tokens, parent, T, V, path_len, out_tokens,
                     path_nodes, stream=None) -> None:
    _call("spec_accept_tree", _h(ctx), _ptr(target_logits), _ptr(draft_tokens), _ptr(parent), T, V,
          _ptr(path_len), _ptr(out_tokens), _ptr(path_nodes), _stream(stream))


def spec_gumbel_sample(ctx, logits, rows, V, seed, position, out_tokens, near_tie_flags=None,
                       stream=None) -> None:
    _call("spec_gumbel_sample", _h(ctx), _ptr(logits), rows, V, seed % (1 << 64), position % (1 << 64),
          _ptr(out_tokens), _ptr(near_tie_flags), _stream(stream))


def spec_accept_gumbel(ctx, target_logits, draft_tokens, T, V, seed, position, n_accepted,
                       out_tokens, near_tie_flags=None, stream=None) -> None:
    _call("spec_accept_gumbel", _h(ctx), _ptr(target_logits), _ptr(draft_tokens), T, V,
          seed % (1 << 64), position % (1 << 64), _ptr(n_accepted), _ptr(out_tokens),
          _ptr(near_tie_flags), _stream(stream))


def qdequant_w4(ctx, qcodes, scales, zeros, group_size, N, K, w, stream=None) -> None:
    _call("qdequant_w4", _h(ctx), _ptr(qcodes), _ptr(scales), _ptr(zeros), group_size, N, K,
          _ptr(w), _stream(stream))


def qdequant_w8(ctx, qcodes, scales, group_size, N, K, w, stream=None) -> None:
    _call("qdequant_w8", _h(ctx), _ptr(qcodes), _ptr(scales), group_size, N, K, _ptr(w),
          _stream(stream))


def spec_repack_w4_codes(src, dst, N: int, K: int) -> None:
    """Host arrays (numpy uint8, C-contiguous, N*K/2 bytes each); dst may be src."""
    for a in (src, dst):
        if not (a.flags["C_CONTIGUOUS"] and a.dtype.itemsize == 1 and a.size == N * K // 2):
            raise ValueError("src and dst must be C-contiguous byte arrays of N*K/2 bytes")
    _call("spec_repack_w4_codes", src.ctypes.data, dst.ctypes.data, N, K)
