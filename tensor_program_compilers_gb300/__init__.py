"""GB300 fused attention forward: Python binding of libattn's C ABI.

The compute lives in ``csrc/attn_fwd.cu`` (sm_103a: TMA, mbarriers, tcgen05
MMAs accumulating in tensor memory); ``include/attn.h`` documents the ABI.
This module only marshals arguments: it passes device pointers, sizes and the
current CUDA stream to the shared library and turns status codes into
exceptions.  There is no fallback: if ``libattn.so`` is missing or the device
is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
LIB_PATH = os.path.join(_HERE, "libattn.so")
INCLUDE_DIR = os.path.join(_ROOT, "include")
SOURCES = [os.path.join(_CSRC, "attn_fwd.cu")]
DEPENDS = SOURCES + [os.path.join(_CSRC, "ptx.cuh"), os.path.join(_CSRC, "attn_bwd.cuh"),
                     os.path.join(_CSRC, "attn_fwd2.cuh"), os.path.join(_CSRC, "attn_bwd256.cuh"),
                     os.path.join(_CSRC, "attn_decode_cc.cuh"),
                     os.path.join(_CSRC, "attn_bwd_fused.cuh"),
                     os.path.join(INCLUDE_DIR, "attn.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]

# status codes (include/attn.h)
ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_ALIGNMENT = 2
ATTN_ERR_UNSUPPORTED_DEVICE = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_BAD_SEQLENS = 6
ATTN_ERR_BAD_PAGE_TABLE = 7

EXPORTED = ["attn_fwd", "attn_fwd_ex", "attn_fwd_decode", "attn_decode_workspace_bytes",
            "attn_fwd_decode_paged", "attn_decode_paged_workspace_bytes",
            "attn_fwd_decode_static", "attn_bwd", "attn_bwd_workspace_bytes",
            "attn_bwd_single_pass", "attn_bwd_single_pass_workspace_bytes",
            "attn_get_status", "attn_status_string", "attn_selftest_timeout",
            "attn_debug_one_tile", "attn_probe_dram_latency"]


class AttnVariant(ctypes.Structure):
    """``attn_variant`` of include/attn.h: key window, soft cap, ALiBi slopes."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("softcap", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p)]


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {attn_status_string(code)} ({code})")
        self.code = code


def nvcc_path() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libattn.so in-tree for sm_103a (skipped when up to date)."""
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(p) for p in DEPENDS)):
        return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc_path(), *NVCC_FLAGS, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True, timeout=900)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libattn.so is not built ({LIB_PATH}); run tensor_program_compilers_gb300.build()")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.attn_fwd.restype = i
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp, vp]
        lib.attn_fwd_ex.restype = i
        lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp,
                                    ctypes.POINTER(AttnVariant), vp]
        lib.attn_fwd_decode.restype = i
        lib.attn_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i,
                                        vp, vp, ctypes.c_size_t, vp]
        lib.attn_fwd_decode_static.restype = i
        lib.attn_fwd_decode_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                               ctypes.c_float, i, vp, vp]
        lib.attn_fwd_decode_paged.restype = i
        lib.attn_fwd_decode_paged.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i,
                                              vp, vp, i, i, i, vp, ctypes.c_size_t, vp]
        lib.attn_decode_paged_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_decode_paged_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.attn_bwd.restype = i
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                 ctypes.c_float, i, vp, vp, ctypes.c_size_t, vp]
        lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.attn_bwd_single_pass.restype = i
        lib.attn_bwd_single_pass.argtypes = lib.attn_bwd.argtypes
        lib.attn_bwd_single_pass_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd_single_pass_workspace_bytes.argtypes = [i, i, i, i]
        lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.attn_get_status.restype = i
        lib.attn_get_status.argtypes = [vp]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_status_string.argtypes = [i]
        lib.attn_selftest_timeout.restype = i
        lib.attn_selftest_timeout.argtypes = [i, vp]
        lib.attn_debug_one_tile.restype = i
        lib.attn_debug_one_tile.argtypes = [i]
        lib.attn_probe_dram_latency.restype = i
        lib.attn_probe_dram_latency.argtypes = [vp, ctypes.c_size_t, i, vp, vp]
        _lib = lib
    return _lib


def library():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_status_string(code: int) -> str:
    return _load().attn_status_string(int(code)).decode()


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, cu_seqlens=None,
             stream=None, check=True) -> int:
    """Call the C ``attn_fwd`` with device tensors (or raw device pointers).

    Layouts and argument meaning are those of ``include/attn.h``.  Returns
    the status code; with ``check`` a non-OK code raises AttnError.
    """
    rc = _load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                          int(Hkv), int(N), int(d), float(scale), int(bool(causal)),
                          _ptr(cu_seqlens), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return rc


def make_variant(window=None, softcap: float = 0.0, alibi_slopes=None) -> AttnVariant:
    """window = (left, right) key bounds around each row (None or a negative
    side: unbounded); softcap > 0 caps scaled scores at +-softcap via tanh;
    alibi_slopes: device fp32 tensor [Hq] (or a raw pointer) or None."""
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    return AttnVariant(wl, wr, float(softcap), _ptr(alibi_slopes))


def attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, cu_seqlens=None,
                window=None, softcap=0.0, alibi_slopes=None, stream=None, check=True) -> int:
    """Call the C ``attn_fwd_ex`` (attn_fwd plus the score and mask variants)."""
    var = make_variant(window, softcap, alibi_slopes)
    rc = _load().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                             int(Hkv), int(N), int(d), float(scale), int(bool(causal)),
                             _ptr(cu_seqlens), ctypes.byref(var), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_ex")
    return rc


def attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d) -> int:
    """Workspace bytes ``attn_fwd_decode`` needs on the current device."""
    return int(_load().attn_decode_workspace_bytes(int(B), int(Hq), int(Hkv), int(Nq), int(Nk),
                                                   int(d)))


def attn_fwd_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, seqlens_k=None,
                    workspace=None, workspace_bytes=None, stream=None, check=True) -> int:
    """Call the C ``attn_fwd_decode`` (split-key attention for decode shapes).

    q, o [B, Nq, Hq, d]; k, v [B, Nk, Hkv, d]; lse [B, Hq, Nq]; seqlens_k
    int32 [B] on the device or None; workspace: a device buffer of at least
    ``attn_decode_workspace_bytes`` bytes (a tensor, or a raw pointer with
    workspace_bytes).
    """
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = _load().attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                                 int(Hkv), int(Nq), int(Nk), int(d), float(scale),
                                 int(bool(causal)), _ptr(seqlens_k), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_decode")
    return rc


def attn_decode_paged_workspace_bytes(B, Hq, Hkv, Nq, max_blocks, page_size, d) -> int:
    """Workspace bytes ``attn_fwd_decode_paged`` needs on the current device."""
    return int(_load().attn_decode_paged_workspace_bytes(int(B), int(Hq), int(Hkv), int(Nq),
                                                         int(max_blocks), int(page_size), int(d)))


def attn_fwd_decode_paged(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nq, d, scale, causal,
                          seqlens_k, block_table, max_blocks, page_size, num_pages,
                          workspace=None, workspace_bytes=None, stream=None, check=True) -> int:
    """Call the C ``attn_fwd_decode_paged``: decode over paged caches
    k_cache, v_cache [num_pages, page_size, Hkv, d] addressed through
    block_table [B, max_blocks] (int32, device) and seqlens_k [B]."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = _load().attn_fwd_decode_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv),
        int(Nq), int(d), float(scale), int(bool(causal)), _ptr(seqlens_k), _ptr(block_table),
        int(max_blocks), int(page_size), int(num_pages), _ptr(workspace), int(workspace_bytes),
        _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_decode_paged")
    return rc


def attn_bwd_workspace_bytes(B, Hq, N, packed=False) -> int:
    """Workspace bytes ``attn_bwd`` needs (per-row D and LSE, sequence offsets)."""
    return int(_load().attn_bwd_workspace_bytes(int(B), int(Hq), int(N), int(bool(packed))))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal,
             cu_seqlens=None, workspace=None, workspace_bytes=None, stream=None,
             check=True) -> int:
    """Call the C ``attn_bwd``: dq, dk, dv of the forward's O for output
    gradient dout (the forward's layouts and LSE; packed with cu_seqlens)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = _load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(N), int(d),
                          float(scale), int(bool(causal)), _ptr(cu_seqlens), _ptr(workspace),
                          int(workspace_bytes), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return rc


def attn_bwd_single_pass_workspace_bytes(B, Hq, N, packed=False) -> int:
    """Workspace bytes ``attn_bwd_single_pass`` needs (the fp32 dQ buffer,
    then ``attn_bwd``'s)."""
    return int(_load().attn_bwd_single_pass_workspace_bytes(int(B), int(Hq), int(N),
                                                            int(bool(packed))))


def attn_bwd_single_pass(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal,
                         cu_seqlens=None, workspace=None, workspace_bytes=None, stream=None,
                         check=True) -> int:
    """Call the C ``attn_bwd_single_pass`` (d = 64): arguments as ``attn_bwd``."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = _load().attn_bwd_single_pass(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        int(B), int(Hq), int(Hkv), int(N), int(d), float(scale), int(bool(causal)),
        _ptr(cu_seqlens), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_single_pass")
    return rc


def attention_backward(q, k, v, o, lse, dout, causal: bool, scale: Optional[float] = None,
                       cu_seqlens=None, stream=None, single_pass: bool = False):
    """Allocate dq, dk, dv and the workspace (torch, on q's device) and run
    ``attn_bwd`` (or, single_pass and d = 64, ``attn_bwd_single_pass``):
    fixed batch q [B, N, Hq, d], k/v [B, N, Hkv, d], or packed q [T, Hq, d],
    k/v [T, Hkv, d] with cu_seqlens (int32 [B+1], device)."""
    import torch
    d = q.shape[-1]
    if cu_seqlens is None:
        B, N, Hq, _ = q.shape
        Hkv = k.shape[2]
    else:
        N, Hq, _ = q.shape
        Hkv = k.shape[1]
        B = cu_seqlens.numel() - 1
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    size = attn_bwd_single_pass_workspace_bytes if single_pass else attn_bwd_workspace_bytes
    n = size(B, Hq, N, packed=cu_seqlens is not None)
    ws = torch.empty(((max(n, 16) + 15) // 16 * 4,), dtype=torch.float32, device=q.device)
    run = attn_bwd_single_pass if single_pass else attn_bwd
    run(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, cu_seqlens, ws,
        stream=stream)
    return dq, dk, dv


DECODE_STATIC_SCRATCH_BYTES = 8 << 20


def attn_fwd_decode_static(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, seqlens_k=None,
                           stream=None, check=True) -> int:
    """Call the C ``attn_fwd_decode_static``: attn_fwd_decode with the
    library's fixed 8 MiB scratch instead of a workspace (no allocation;
    overlapping calls on one device race)."""
    rc = _load().attn_fwd_decode_static(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                        int(Hq), int(Hkv), int(Nq), int(Nk), int(d),
                                        float(scale), int(bool(causal)), _ptr(seqlens_k),
                                        _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_decode_static")
    return rc


def decode(q, k, v, causal: bool = False, scale: Optional[float] = None, seqlens_k=None,
           out=None, lse=None, workspace=None, stream=None):
    """Allocate outputs and workspace (torch, on q's device) and run
    ``attn_fwd_decode``: q [B, Nq, Hq, d], k/v caches [B, Nk, Hkv, d]."""
    import torch
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    scale = d ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
        workspace = torch.empty((max(n, 16) + 15) // 16 * 4, dtype=torch.float32, device=q.device)
    attn_fwd_decode(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, seqlens_k,
                    workspace, stream=stream)
    return out, lse


def attn_get_status(stream=None) -> int:
    """Take and clear the device status word (one atomic exchange ordered on
    the stream), then synchronise the stream."""
    return _load().attn_get_status(_stream(stream))


def attn_selftest_timeout(timeout_us: int = 1000, stream=None) -> int:
    return _load().attn_selftest_timeout(int(timeout_us), _stream(stream))


def attn_probe_dram_latency(scratch, nbytes: int, hops: int, result, stream=None,
                            check=True) -> int:
    """Call the C ``attn_probe_dram_latency``: chase ``hops`` links of a chain
    written into ``scratch`` (device, ``nbytes``); ``result`` (device, two
    uint64 words) receives the chase's nanoseconds and the final index."""
    rc = _load().attn_probe_dram_latency(_ptr(scratch), int(nbytes), int(hops), _ptr(result),
                                         _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_probe_dram_latency")
    return rc


def attn_debug_one_tile(on: bool) -> bool:
    """Route every later forward through the one-tile kernel (tests); returns
    the previous setting."""
    return bool(_load().attn_debug_one_tile(1 if on else 0))


def attention(q, k, v, causal: bool, scale: Optional[float] = None, cu_seqlens=None,
              out=None, lse=None, stream=None, window=None, softcap: float = 0.0,
              alibi_slopes=None):
    """Allocate outputs (torch, on q's device) and run ``attn_fwd_ex``.

    Fixed batch: q [B, N, Hq, d], k/v [B, N, Hkv, d] -> o like q, lse [B, Hq, N].
    Packed: q [T, Hq, d], k/v [T, Hkv, d], cu_seqlens int32 [B+1] on the
    device -> o like q, lse [Hq, T].  window / softcap / alibi_slopes: the
    score and mask variants (see ``make_variant``).
    """
    import torch
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    if cu_seqlens is None:
        B, N, Hq, _ = q.shape
        Hkv = k.shape[2]
        lse_shape = (B, Hq, N)
        n_arg = N
    else:
        T, Hq, _ = q.shape
        Hkv = k.shape[1]
        B = cu_seqlens.numel() - 1
        lse_shape = (Hq, T)
        n_arg = T
    for t in (q, k, v):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    attn_fwd_ex(q, k, v, out, lse, B, Hq, Hkv, n_arg, d, scale, causal, cu_seqlens,
                window=window, softcap=softcap, alibi_slopes=alibi_slopes, stream=stream)
    return out, lse
