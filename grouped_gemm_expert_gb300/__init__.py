"""Python binding of the K-grouped MoE weight-gradient library (``libkgw.so``).

Argument marshalling only: every step of the operation runs in the CUDA kernels of the
shared library. PyTorch supplies device memory and streams. There is no fallback: if the
library has not been built (``python -m grouped_gemm_expert_gb300.build``) or the device is
not sm_103, calls raise.

The functions keep the C names of ``include/kgw.h``:

  kgw_workspace_size(args, is_fp8) -> int
  kgw_wgrad_bf16(args, workspace, stream=None)
  kgw_wgrad_fp8_blockscaled(args, sfa, sfb, workspace, stream=None)
  kgw_status_string(code) -> str
  kgw_version() -> int
  kgw_debug_set(key, value) -> int
  kgw_wgrad_bf16_noalloc(args, stream=None)
  kgw_debug_check_ragged_maps(args, is_fp8, host_offsets, workspace) -> int
  kgw_wgrad_fp8_ue8m0(args, sfa_packed, sfb_packed, workspace, stream=None)
  kgw_wgrad_fp4_ue8m0(args, sfa_packed, sfb_packed, workspace, stream=None)
  kgw_wgrad_bf16_unaligned(args, workspace, stream=None)
  kgw_mgrouped_workspace_size(args) -> int
  kgw_mgrouped_bf16(args, workspace, stream=None)
  kgw_mgrouped_fp8(args, sfa, sfb, sf_format, workspace, stream=None)
  kgw_wgrad_nvfp4(args, sfa_packed, sfb_packed, global_scale_a, global_scale_b, workspace, stream=None)
  kgw_wgrad_fp8_unaligned(args, sfa, sfb, sf_format, workspace, stream=None)
  kgw_wgrad_fp4_unaligned(args, sfa_packed, sfb_packed, workspace, stream=None)
  kgw_debug_check_tail_maps_kind(args, kind, host_offsets, workspace) -> int

``make_args`` / ``make_mgrouped_args`` build the argument structs from torch tensors.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkgw.so")

KGW_OK = 0
KGW_ERR_INVALID_ARG = 1
KGW_ERR_UNSUPPORTED = 2
KGW_ERR_ALIGNMENT = 3
KGW_ERR_DEVICE = 4
KGW_ERR_CUDA = 5
KGW_ERR_OFFSETS = 6
KGW_ERR_TIMEOUT = 7
KGW_ERR_WORKSPACE = 8
KGW_ERR_OUT_PTRS = 9
KGW_ERR_SCRATCH_LIMIT = 10
KGW_ERR_SCALES = 11

KGW_K_MAJOR = 0
KGW_MN_MAJOR = 1
KGW_TENSOR2D = 0
KGW_RAGGED = 1
KGW_OUT_F32 = 0
KGW_OUT_BF16 = 1
KGW_OUT_F16 = 2
KGW_MG_OFFSETS = 0
KGW_MG_INDICES = 1
KGW_MG_MASKED = 2

EXPORTED = ("kgw_workspace_size", "kgw_wgrad_bf16", "kgw_wgrad_fp8_blockscaled",
            "kgw_status_string", "kgw_version", "kgw_debug_set", "kgw_wgrad_bf16_noalloc",
            "kgw_debug_check_ragged_maps", "kgw_wgrad_fp8_ue8m0", "kgw_mgrouped_workspace_size",
            "kgw_mgrouped_bf16", "kgw_wgrad_fp4_ue8m0", "kgw_wgrad_bf16_unaligned",
            "kgw_debug_check_tail_maps", "kgw_mgrouped_fp8", "kgw_wgrad_fp8_unaligned", "kgw_wgrad_fp4_unaligned",
            "kgw_debug_check_tail_maps_kind", "kgw_wgrad_nvfp4")


class KgwArgs(ctypes.Structure):
    """Mirror of ``kgw_wgrad_args`` (include/kgw.h)."""
    _fields_ = [
        ("num_experts", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("intermediate", ctypes.c_int32),
        ("tokens_sum", ctypes.c_int64),
        ("a", ctypes.c_void_p),
        ("a_major", ctypes.c_int32),
        ("b", ctypes.c_void_p),
        ("b_major", ctypes.c_int32),
        ("offsets", ctypes.c_void_p),
        ("input_order", ctypes.c_int32),
        ("out", ctypes.c_void_p),
        ("out_ptrs", ctypes.c_void_p),
        ("out_dtype", ctypes.c_int32),
        ("accumulate", ctypes.c_int32),
        ("status_dev", ctypes.c_void_p),
    ]


class KgwMgroupedArgs(ctypes.Structure):
    """Mirror of ``kgw_mgrouped_args`` (include/kgw.h)."""
    _fields_ = [
        ("num_groups", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("m", ctypes.c_int64),
        ("n", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("a", ctypes.c_void_p),
        ("b", ctypes.c_void_p),
        ("b_major", ctypes.c_int32),
        ("groups", ctypes.c_void_p),
        ("d", ctypes.c_void_p),
        ("out_dtype", ctypes.c_int32),
        ("accumulate", ctypes.c_int32),
        ("status_dev", ctypes.c_void_p),
    ]


class KgwError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {kgw_status_string(code)} ({code})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libkgw.so`` (raises if it is missing: there is no other implementation)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run `python -m grouped_gemm_expert_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.kgw_workspace_size.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
        L.kgw_workspace_size.restype = ctypes.c_int
        L.kgw_wgrad_bf16.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_wgrad_bf16.restype = ctypes.c_int
        L.kgw_wgrad_fp8_blockscaled.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_wgrad_fp8_blockscaled.restype = ctypes.c_int
        L.kgw_wgrad_fp8_ue8m0.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_wgrad_fp8_ue8m0.restype = ctypes.c_int
        L.kgw_wgrad_fp4_ue8m0.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_wgrad_fp4_ue8m0.restype = ctypes.c_int
        L.kgw_wgrad_bf16_unaligned.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_size_t,
                                               ctypes.c_void_p]
        L.kgw_wgrad_bf16_unaligned.restype = ctypes.c_int
        L.kgw_mgrouped_workspace_size.argtypes = [ctypes.POINTER(KgwMgroupedArgs), ctypes.POINTER(ctypes.c_size_t)]
        L.kgw_mgrouped_workspace_size.restype = ctypes.c_int
        L.kgw_mgrouped_bf16.argtypes = [ctypes.POINTER(KgwMgroupedArgs), ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p]
        L.kgw_mgrouped_bf16.restype = ctypes.c_int
        L.kgw_mgrouped_fp8.argtypes = [ctypes.POINTER(KgwMgroupedArgs), ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_mgrouped_fp8.restype = ctypes.c_int
        L.kgw_status_string.argtypes = [ctypes.c_int32]
        L.kgw_status_string.restype = ctypes.c_char_p
        L.kgw_version.argtypes = []
        L.kgw_version.restype = ctypes.c_int32
        L.kgw_wgrad_bf16_noalloc.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p]
        L.kgw_wgrad_bf16_noalloc.restype = ctypes.c_int
        L.kgw_debug_check_ragged_maps.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_int32, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_debug_check_ragged_maps.restype = ctypes.c_int32
        L.kgw_debug_check_tail_maps.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_debug_check_tail_maps.restype = ctypes.c_int32
        L.kgw_wgrad_nvfp4.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_wgrad_nvfp4.restype = ctypes.c_int
        L.kgw_wgrad_fp8_unaligned.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_wgrad_fp8_unaligned.restype = ctypes.c_int
        L.kgw_wgrad_fp4_unaligned.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_wgrad_fp4_unaligned.restype = ctypes.c_int
        L.kgw_debug_check_tail_maps_kind.argtypes = [ctypes.POINTER(KgwArgs), ctypes.c_int32, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.kgw_debug_check_tail_maps_kind.restype = ctypes.c_int32
        L.kgw_debug_set.argtypes = [ctypes.c_int32, ctypes.c_int64]
        L.kgw_debug_set.restype = ctypes.c_int64
        _lib = L
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def make_args(num_experts: int, hidden: int, intermediate: int, tokens_sum: int, a, b, offsets, *,
              out=None, out_ptrs=None, out_dtype: int = KGW_OUT_F32, accumulate: bool = False,
              input_order: int = KGW_TENSOR2D, a_major: int = KGW_K_MAJOR, b_major: int = KGW_MN_MAJOR,
              status_dev=None) -> KgwArgs:
    """Build ``kgw_wgrad_args``; tensors (or raw integer addresses) are passed by address."""
    return KgwArgs(num_experts, hidden, intermediate, tokens_sum, _ptr(a), a_major, _ptr(b), b_major,
                   _ptr(offsets), input_order, _ptr(out), _ptr(out_ptrs), out_dtype, int(bool(accumulate)),
                   _ptr(status_dev))


def make_mgrouped_args(num_groups: int, m: int, n: int, k: int, a, b, groups, d, *,
                       layout: int = KGW_MG_OFFSETS, b_major: int = KGW_K_MAJOR, out_dtype: int = KGW_OUT_BF16,
                       accumulate: bool = False, status_dev=None) -> KgwMgroupedArgs:
    """Build ``kgw_mgrouped_args``; tensors (or raw integer addresses) are passed by address."""
    return KgwMgroupedArgs(num_groups, layout, m, n, k, _ptr(a), _ptr(b), b_major, _ptr(groups), _ptr(d),
                           out_dtype, int(bool(accumulate)), _ptr(status_dev))


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kgw_status_string(code: int) -> str:
    return lib().kgw_status_string(int(code)).decode()


def kgw_version() -> int:
    return int(lib().kgw_version())


def kgw_debug_set(key: int, value: int) -> int:
    return int(lib().kgw_debug_set(int(key), int(value)))


def kgw_workspace_size(args: KgwArgs, is_fp8: bool = False) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().kgw_workspace_size(ctypes.byref(args), int(bool(is_fp8)), ctypes.byref(n))
    if rc != KGW_OK:
        raise KgwError(rc, "kgw_workspace_size")
    return int(n.value)


def kgw_wgrad_bf16(args: KgwArgs, workspace, workspace_bytes: Optional[int] = None, stream=None,
                   check: bool = True) -> int:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_bf16(ctypes.byref(args), _ptr(workspace), nbytes, _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_bf16")
    return rc


def kgw_wgrad_bf16_unaligned(args: KgwArgs, workspace, workspace_bytes: Optional[int] = None, stream=None,
                             check: bool = True) -> int:
    """kgw_wgrad_bf16 with token counts that are multiples of 8 (any count if A and B are MN-major)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_bf16_unaligned(ctypes.byref(args), _ptr(workspace), nbytes, _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_bf16_unaligned")
    return rc


def kgw_wgrad_fp8_blockscaled(args: KgwArgs, sfa, sfb, workspace, workspace_bytes: Optional[int] = None,
                              stream=None, check: bool = True) -> int:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_fp8_blockscaled(ctypes.byref(args), _ptr(sfa), _ptr(sfb), _ptr(workspace), nbytes,
                                         _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_fp8_blockscaled")
    return rc


def kgw_wgrad_fp8_ue8m0(args: KgwArgs, sfa_packed, sfb_packed, workspace, workspace_bytes: Optional[int] = None,
                        stream=None, check: bool = True) -> int:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_fp8_ue8m0(ctypes.byref(args), _ptr(sfa_packed), _ptr(sfb_packed), _ptr(workspace), nbytes,
                                   _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_fp8_ue8m0")
    return rc


def kgw_wgrad_nvfp4(args: KgwArgs, sfa_packed, sfb_packed, global_scale_a, global_scale_b, workspace,
                    workspace_bytes: Optional[int] = None, stream=None, check: bool = True) -> int:
    """NVFP4: e2m1 operands (K-major), UE4M3 scales per 16 tokens packed four to an int32 word, and
    per-tensor FP32 global scales given as device tensors of one float (or None for 1)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_nvfp4(ctypes.byref(args), _ptr(sfa_packed), _ptr(sfb_packed), _ptr(global_scale_a),
                               _ptr(global_scale_b), _ptr(workspace), nbytes, _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_nvfp4")
    return rc


def kgw_wgrad_fp8_unaligned(args: KgwArgs, sfa, sfb, sf_format: int, workspace,
                            workspace_bytes: Optional[int] = None, stream=None, check: bool = True) -> int:
    """FP8 with token counts that are multiples of 16 (any count if A and B are MN-major); scales
    per 128-token block of each expert, sf_format 0 (FP32) or 1 (packed UE8M0 per 32 tokens)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_fp8_unaligned(ctypes.byref(args), _ptr(sfa), _ptr(sfb), int(sf_format), _ptr(workspace),
                                       nbytes, _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_fp8_unaligned")
    return rc


def kgw_wgrad_fp4_unaligned(args: KgwArgs, sfa_packed, sfb_packed, workspace, workspace_bytes: Optional[int] = None,
                            stream=None, check: bool = True) -> int:
    """FP4 (K-major A and B) with token counts that are multiples of 32; packed UE8M0 scales per
    32 tokens of each expert's 128-token blocks."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_fp4_unaligned(ctypes.byref(args), _ptr(sfa_packed), _ptr(sfb_packed), _ptr(workspace),
                                       nbytes, _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_fp4_unaligned")
    return rc


def kgw_mgrouped_workspace_size(args: KgwMgroupedArgs) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().kgw_mgrouped_workspace_size(ctypes.byref(args), ctypes.byref(n))
    if rc != KGW_OK:
        raise KgwError(rc, "kgw_mgrouped_workspace_size")
    return int(n.value)


def kgw_mgrouped_bf16(args: KgwMgroupedArgs, workspace, workspace_bytes: Optional[int] = None, stream=None,
                      check: bool = True) -> int:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_mgrouped_bf16(ctypes.byref(args), _ptr(workspace), nbytes, _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_mgrouped_bf16")
    return rc


def kgw_wgrad_fp4_ue8m0(args: KgwArgs, sfa_packed, sfb_packed, workspace, workspace_bytes: Optional[int] = None,
                        stream=None, check: bool = True) -> int:
    """FP4 e2m1 operands (packed uint8, K-major A and B) with packed UE8M0 scales per 32 tokens."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_wgrad_fp4_ue8m0(ctypes.byref(args), _ptr(sfa_packed), _ptr(sfb_packed), _ptr(workspace), nbytes,
                                   _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_fp4_ue8m0")
    return rc


def kgw_mgrouped_fp8(args: KgwMgroupedArgs, sfa, sfb, sf_format: int, workspace,
                     workspace_bytes: Optional[int] = None, stream=None, check: bool = True) -> int:
    """FP8 M-grouped GEMM: e4m3 operands, sf_format 0 (FP32 per 128 K) or 1 (packed UE8M0 per 32 K)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib().kgw_mgrouped_fp8(ctypes.byref(args), _ptr(sfa), _ptr(sfb), int(sf_format), _ptr(workspace), nbytes,
                                _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_mgrouped_fp8")
    return rc


def kgw_wgrad_bf16_noalloc(args: KgwArgs, stream=None, check: bool = True) -> int:
    """kgw_wgrad_bf16 using the library's static 2 MiB scratch instead of a workspace.

    For callers that cannot allocate device memory when they call (see include/kgw.h). The
    first call on a device performs a one-time set-up and should precede any stream capture;
    calls that overlap on the GPU share the scratch and must be ordered.
    """
    rc = lib().kgw_wgrad_bf16_noalloc(ctypes.byref(args), _stream_handle(stream))
    if check and rc != KGW_OK:
        raise KgwError(rc, "kgw_wgrad_bf16_noalloc")
    return rc


def kgw_debug_check_ragged_maps(args: KgwArgs, is_fp8: bool, host_offsets, workspace,
                                workspace_bytes: Optional[int] = None, host_dump=None) -> int:
    """Testing hook: number of experts whose device-built A descriptor differs from the host encoding."""
    import numpy as np
    offs = np.ascontiguousarray(np.asarray(host_offsets, dtype=np.int32))
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    dump = None if host_dump is None else host_dump.ctypes.data
    return int(lib().kgw_debug_check_ragged_maps(ctypes.byref(args), int(bool(is_fp8)), offs.ctypes.data,
                                                 _ptr(workspace), nbytes, dump))


def kgw_debug_check_tail_maps(args: KgwArgs, host_offsets, workspace, workspace_bytes: Optional[int] = None,
                              host_dump=None) -> int:
    """Testing hook: number of per-expert token-tail descriptors that differ from host encodings."""
    import numpy as np
    offs = np.ascontiguousarray(np.asarray(host_offsets, dtype=np.int32))
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    dump = None if host_dump is None else host_dump.ctypes.data
    return int(lib().kgw_debug_check_tail_maps(ctypes.byref(args), offs.ctypes.data, _ptr(workspace), nbytes, dump))


def kgw_debug_check_tail_maps_kind(args: KgwArgs, kind: int, host_offsets, workspace,
                                   workspace_bytes: Optional[int] = None, host_dump=None) -> int:
    """Testing hook: kgw_debug_check_tail_maps for BF16 (kind 0), FP8 (1) or FP4 (2) descriptors."""
    import numpy as np
    offs = np.ascontiguousarray(np.asarray(host_offsets, dtype=np.int32))
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    dump = None if host_dump is None else host_dump.ctypes.data
    return int(lib().kgw_debug_check_tail_maps_kind(ctypes.byref(args), int(kind), offs.ctypes.data,
                                                    _ptr(workspace), nbytes, dump))


# ---------------------------------------------------------------------------------------------
# Convenience layer over torch tensors (still marshalling only)
# ---------------------------------------------------------------------------------------------

def workspace_for(args: KgwArgs, is_fp8: bool = False, device=None):
    import torch
    n = kgw_workspace_size(args, is_fp8)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def wgrad(a, b, offsets, *, hidden: int, intermediate: int, out=None, out_ptrs=None,
          out_dtype: str = "f32", accumulate: bool = False, input_order: str = "tensor2d",
          sfa=None, sfb=None, workspace=None, status_dev=None, stream=None):
    """One call of the operation on torch CUDA tensors. ``a``/``b`` are bf16 or float8_e4m3fn.

    Exactly one of ``out`` (dense [E, hidden, intermediate]) and ``out_ptrs`` (int64 [E]
    device addresses) must be given. Returns ``out`` (or None for pointer outputs).
    """
    import torch
    E = int(offsets.numel())
    tokens_sum = int(b.shape[0]) if b.dim() == 2 else 0
    fp8 = a.dtype == torch.float8_e4m3fn
    args = make_args(E, hidden, intermediate, tokens_sum, a, b, offsets, out=out, out_ptrs=out_ptrs,
                     out_dtype={"bf16": KGW_OUT_BF16, "f16": KGW_OUT_F16}.get(out_dtype, KGW_OUT_F32),
                     accumulate=accumulate, input_order=KGW_RAGGED if input_order == "ragged" else KGW_TENSOR2D,
                     status_dev=status_dev)
    if workspace is None:
        workspace = workspace_for(args, fp8, device=b.device)
    if fp8:
        kgw_wgrad_fp8_blockscaled(args, sfa, sfb, workspace, stream=stream)
    else:
        kgw_wgrad_bf16(args, workspace, stream=stream)
    return out


def mgrouped(a, b, groups, *, layout: str = "offsets", d=None, b_major: str = "k", out_dtype: str = "bf16",
             accumulate: bool = False, workspace=None, status_dev=None, stream=None, sfa=None, sfb=None,
             sf_format: str = "f32_128"):
    """M-grouped GEMM on torch CUDA tensors: D[rows of g] (+)= A[rows of g] @ op(B[g]).

    ``a`` bf16 [m, k] (contiguous layouts) or [G, max_m, k] (``layout="masked"``); ``b`` bf16
    [G, n, k] (``b_major="k"``, op = transpose) or [G, k, n] (``b_major="mn"``); ``groups`` int32:
    cumulative row counts [G] (``"offsets"``), per-row group ids [m] (``"indices"``) or valid rows
    per group [G] (``"masked"``). Returns ``d``.
    """
    import torch
    G = int(b.shape[0])
    k = int(a.shape[-1])
    m = int(a.shape[1] if layout == "masked" else a.shape[0])
    n = int(b.shape[1] if b_major == "k" else b.shape[2])
    lay = {"offsets": KGW_MG_OFFSETS, "indices": KGW_MG_INDICES, "masked": KGW_MG_MASKED}[layout]
    odt = {"bf16": KGW_OUT_BF16, "f16": KGW_OUT_F16, "f32": KGW_OUT_F32}[out_dtype]
    if d is None:
        shape = (G, m, n) if layout == "masked" else (m, n)
        d = torch.zeros(shape, dtype={"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[out_dtype],
                        device=a.device)
    args = make_mgrouped_args(G, m, n, k, a, b, groups, d, layout=lay,
                              b_major=KGW_K_MAJOR if b_major == "k" else KGW_MN_MAJOR, out_dtype=odt,
                              accumulate=accumulate, status_dev=status_dev)
    if workspace is None:
        workspace = torch.empty(kgw_mgrouped_workspace_size(args), dtype=torch.uint8, device=a.device)
    if a.dtype == torch.float8_e4m3fn:
        kgw_mgrouped_fp8(args, sfa, sfb, 1 if sf_format == "ue8m0_32" else 0, workspace, stream=stream)
    else:
        kgw_mgrouped_bf16(args, workspace, stream=stream)
    return d
