"""Thin Python binding of libmoelora.so (ctypes): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module checks tensor
dtypes/devices/contiguity, passes raw device pointers and the current CUDA stream, and
turns status codes into exceptions.  PyTorch provides device memory and streams.
If the library has not been built, every call raises MoELoRAError: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoelora.so")

MOE_LORA_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE_TOO_SMALL", 4: "CUDA",
                5: "TIMEOUT", 6: "DEVICE_CHECK"}
ROUTE_RENORMALIZE = 0
ROUTE_DEEPSEEK_V3 = 1
FLAG_LORA_OFF = 1
FLAG_FORCE_SINGLE_STREAM = 2
FLAG_FORCE_TWO_STREAM = 4
FLAG_UNFUSED_LORA = 8
FLAG_NO_PDL = 16
FLAG_SHARED_OUTER = 32
FLAG_DOWN_LORA_SIDE = 64
FLAG_SEPARATE_SHRINK = 128
STAGES = ["route", "permute", "gate_up_gemm", "lora_gate_up", "activation", "down_gemm",
          "lora_down", "finalize"]
NUM_STAGES = len(STAGES)

EXPORTED = ["moe_lora_create", "moe_lora_destroy", "moe_lora_status_string", "moe_lora_last_cuda_error",
            "moe_lora_workspace_size", "moe_lora_validate", "moe_lora_route", "moe_lora_permute",
            "moe_lora_forward", "moe_lora_check_status", "moe_lora_route_noalloc", "moe_lora_forward_routed",
            "moe_lora_launch_count", "moe_lora_forward_fp8", "moe_lora_quant_fp8", "moe_lora_grouped_gemm_fp8",
            "moe_lora_forward_nvfp4", "moe_lora_quant_nvfp4", "moe_lora_grouped_gemm_nvfp4",
            "moe_lora_packed_lora_b_size", "moe_lora_pack_lora_b", "moe_lora_packed_lora_a_size",
            "moe_lora_pack_lora_a"]


class MoELoRAError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {STATUS_NAMES.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


c_int, c_float, c_void_p, c_size_t, c_uint = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint


class Shape(ctypes.Structure):
    _fields_ = [("T", c_int), ("H", c_int), ("I", c_int), ("E", c_int), ("top_k", c_int), ("S", c_int), ("R", c_int)]


class Args(ctypes.Structure):
    _fields_ = [
        ("T", c_int), ("H", c_int), ("I", c_int), ("E", c_int), ("top_k", c_int), ("S", c_int), ("R", c_int),
        ("routing_method", c_int), ("routed_scaling_factor", c_float), ("n_group", c_int), ("topk_group", c_int),
        ("hidden", c_void_p), ("router_logits", c_void_p), ("correction_bias", c_void_p),
        ("w1", c_void_p), ("w2", c_void_p),
        ("lora_A_gu", c_void_p), ("lora_B_gu", c_void_p), ("lora_A_dn", c_void_p), ("lora_B_dn", c_void_p),
        ("slot_idx", c_void_p), ("h_ranks", ctypes.POINTER(ctypes.c_int32)),
        ("h_scalings", ctypes.POINTER(c_float)), ("flags", c_uint),
        ("topk_ids", c_void_p), ("topk_weights", c_void_p), ("expert_offsets", c_void_p),
        ("perm", c_void_p), ("inv_perm", c_void_p), ("prof_events", c_void_p),
        ("lora_B_gu_packed", c_void_p), ("lora_B_dn_packed", c_void_p),
        ("lora_A_gu_packed", c_void_p), ("lora_A_dn_packed", c_void_p),
    ]


class Routed(ctypes.Structure):
    _fields_ = [
        ("packed_topk_ids", c_void_p), ("num_experts", c_int), ("local_expert_offset", c_int),
        ("do_finalize", c_int), ("gemm2_output", c_void_p), ("activation_output", c_void_p),
        ("expert_weights", c_void_p), ("expanded_idx_to_permuted_idx", c_void_p),
    ]


class Fp8Weights(ctypes.Structure):
    _fields_ = [("w1", c_void_p), ("w1_scale", c_void_p), ("w2", c_void_p), ("w2_scale", c_void_p)]


class Nvfp4Weights(ctypes.Structure):
    _fields_ = [("w1", c_void_p), ("w1_sf", c_void_p), ("w1_gs", c_void_p), ("w2", c_void_p), ("w2_sf", c_void_p),
                ("w2_gs", c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoelora.so (raises MoELoRAError if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise MoELoRAError(4, "libmoelora.so not found",
                           f"{LIB_PATH}; build it with routed_moe_expert_gb300._build.build()")
    L = ctypes.CDLL(LIB_PATH)
    L.moe_lora_create.argtypes = [ctypes.POINTER(c_void_p), c_int]
    L.moe_lora_destroy.argtypes = [c_void_p]
    L.moe_lora_status_string.argtypes = [c_int]
    L.moe_lora_status_string.restype = ctypes.c_char_p
    L.moe_lora_last_cuda_error.argtypes = []
    L.moe_lora_last_cuda_error.restype = ctypes.c_char_p
    L.moe_lora_workspace_size.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(c_size_t)]
    L.moe_lora_validate.argtypes = [ctypes.POINTER(Args)]
    L.moe_lora_route.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    L.moe_lora_permute.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]
    L.moe_lora_forward.argtypes = [c_void_p, ctypes.POINTER(Args), c_void_p, c_void_p, c_size_t, c_void_p]
    L.moe_lora_check_status.argtypes = [c_void_p, c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    L.moe_lora_launch_count.argtypes = [c_void_p, ctypes.POINTER(ctypes.c_uint64)]
    L.moe_lora_forward_routed.argtypes = [c_void_p, ctypes.POINTER(Args), ctypes.POINTER(Routed), c_void_p, c_void_p,
                                          c_size_t, c_void_p]
    L.moe_lora_forward_fp8.argtypes = [c_void_p, ctypes.POINTER(Args), ctypes.POINTER(Fp8Weights), c_void_p,
                                       c_void_p, c_size_t, c_void_p]
    L.moe_lora_quant_fp8.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]
    L.moe_lora_grouped_gemm_fp8.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                            c_int, c_int, c_void_p, c_void_p]
    L.moe_lora_forward_nvfp4.argtypes = [c_void_p, ctypes.POINTER(Args), ctypes.POINTER(Nvfp4Weights), c_void_p,
                                         c_void_p, c_size_t, c_void_p]
    L.moe_lora_quant_nvfp4.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p]
    L.moe_lora_grouped_gemm_nvfp4.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                              c_int, c_int, c_int, c_int, c_void_p, c_void_p]
    L.moe_lora_packed_lora_b_size.argtypes = [c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(ctypes.c_int32),
                                              ctypes.POINTER(c_size_t)]
    L.moe_lora_pack_lora_b.argtypes = [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                       ctypes.POINTER(ctypes.c_int32), c_void_p, c_void_p]
    L.moe_lora_packed_lora_a_size.argtypes = [c_int, c_int, c_int, c_int, ctypes.POINTER(ctypes.c_int32),
                                              ctypes.POINTER(c_size_t)]
    L.moe_lora_pack_lora_a.argtypes = [c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                       ctypes.POINTER(ctypes.c_int32), c_void_p, c_void_p]
    for name in EXPORTED:
        if name not in ("moe_lora_status_string", "moe_lora_last_cuda_error"):
            getattr(L, name).restype = c_int
    _lib = L
    return L


def _check(status: int, what: str):
    if status != MOE_LORA_OK:
        detail = lib().moe_lora_last_cuda_error().decode() if status == 4 else ""
        raise MoELoRAError(status, what, detail)


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Handle:
    """Owns a moe_lora_handle (side stream + events).  Create outside graph capture."""

    def __init__(self, device: int = 0):
        h = c_void_p()
        _check(lib().moe_lora_create(ctypes.byref(h), int(device)), "moe_lora_create")
        self._h = h
        self.device = device

    @property
    def ptr(self):
        return self._h

    def launch_count(self) -> int:
        """Kernels launched through this handle so far."""
        n = ctypes.c_uint64()
        _check(lib().moe_lora_launch_count(self._h, ctypes.byref(n)), "moe_lora_launch_count")
        return n.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().moe_lora_destroy(self._h)
            self._h = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_lora_create(device: int = 0) -> Handle:
    return Handle(device)


def moe_lora_status_string(status: int) -> str:
    return lib().moe_lora_status_string(int(status)).decode()


def moe_lora_workspace_size(T, H, I, E, top_k, S=0, R=0) -> int:
    n = c_size_t()
    _check(lib().moe_lora_workspace_size(ctypes.byref(Shape(T, H, I, E, top_k, S, R)), ctypes.byref(n)),
           "moe_lora_workspace_size")
    return n.value


def alloc_workspace(T, H, I, E, top_k, S=0, R=0, device="cuda") -> torch.Tensor:
    return torch.empty(moe_lora_workspace_size(T, H, I, E, top_k, S, R), dtype=torch.uint8, device=device)


def packed_lora_b_shape(E_b: int, N: int, gated: int, ranks: Sequence[int]):
    """Shape of the expand-ready LoRA B copy: (E_b * NT * 128, Rs), NT = N/128 (gated) or
    ceil(N/128), Rs = the sum of the ranks each rounded up to 16 (the C ABI's layout)."""
    NT = N // 128 if gated else (N + 127) // 128
    rs = sum((int(r) + 15) // 16 * 16 for r in ranks if int(r) > 0)
    return (int(E_b) * NT * 128, rs)


def moe_lora_packed_lora_b_size(S, E_b, N, R, gated, ranks) -> int:
    """Bytes of the expand-ready LoRA B copy (host only)."""
    ranks_arr = (ctypes.c_int32 * max(len(ranks), 1))(*[int(r) for r in ranks])
    n = c_size_t(0)
    _check(lib().moe_lora_packed_lora_b_size(int(S), int(E_b), int(N), int(R), int(gated), ranks_arr,
                                             ctypes.byref(n)), "moe_lora_packed_lora_b_size")
    return int(n.value)


def moe_lora_pack_lora_b(handle: Handle, B: torch.Tensor, ranks: Sequence[int], gated: int, out=None,
                         stream=None) -> torch.Tensor:
    """Expand-ready copy of a stacked LoRA B [S, E_b, N, R] (lora_B_gu with gated=1,
    lora_B_dn with gated=0) for the given slot ranks; returns [E_b * NT * 128, Rs] bf16."""
    if B.dim() != 4 or B.dtype != torch.bfloat16 or not B.is_contiguous():
        raise ValueError("B must be a contiguous bf16 [S, E_b, N, R] tensor")
    S, Eb, N, R = (int(x) for x in B.shape)
    if len(ranks) != S:
        raise ValueError(f"need {S} ranks, got {len(ranks)}")
    shape = packed_lora_b_shape(Eb, N, gated, ranks)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=B.device)
    elif tuple(out.shape) != shape:
        raise ValueError(f"out must have shape {shape}")
    ranks_arr = (ctypes.c_int32 * S)(*[int(r) for r in ranks])
    _check(lib().moe_lora_pack_lora_b(handle.ptr, _ptr(B, torch.bfloat16, "B"), S, Eb, N, R, int(gated), ranks_arr,
                                      _ptr(out, torch.bfloat16, "out"), _stream(stream)), "moe_lora_pack_lora_b")
    return out


def packed_lora_a_shape(E_a: int, K: int, ranks: Sequence[int]):
    """Shape of the shrink-ready LoRA A copy: (E_a * RS, K), RS = the sum of the ranks each
    rounded up to 8 (the C ABI's layout)."""
    rs = sum((int(r) + 7) // 8 * 8 for r in ranks if int(r) > 0)
    return (int(E_a) * rs, int(K))


def moe_lora_packed_lora_a_size(S, E_a, K, R, ranks) -> int:
    """Bytes of the shrink-ready LoRA A copy (host only)."""
    ranks_arr = (ctypes.c_int32 * max(len(ranks), 1))(*[int(r) for r in ranks])
    n = c_size_t(0)
    _check(lib().moe_lora_packed_lora_a_size(int(S), int(E_a), int(K), int(R), ranks_arr, ctypes.byref(n)),
           "moe_lora_packed_lora_a_size")
    return int(n.value)


def moe_lora_pack_lora_a(handle: Handle, A: torch.Tensor, ranks: Sequence[int], out=None,
                         stream=None) -> torch.Tensor:
    """Shrink-ready copy of a stacked LoRA A [S, E_a, R, K] for the given slot ranks;
    returns [E_a * RS, K] bf16."""
    if A.dim() != 4 or A.dtype != torch.bfloat16 or not A.is_contiguous():
        raise ValueError("A must be a contiguous bf16 [S, E_a, R, K] tensor")
    S, Ea, R, K = (int(x) for x in A.shape)
    if len(ranks) != S:
        raise ValueError(f"need {S} ranks, got {len(ranks)}")
    shape = packed_lora_a_shape(Ea, K, ranks)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=A.device)
    elif tuple(out.shape) != shape:
        raise ValueError(f"out must have shape {shape}")
    ranks_arr = (ctypes.c_int32 * S)(*[int(r) for r in ranks])
    _check(lib().moe_lora_pack_lora_a(handle.ptr, _ptr(A, torch.bfloat16, "A"), S, Ea, K, R, ranks_arr,
                                      _ptr(out, torch.bfloat16, "out"), _stream(stream)), "moe_lora_pack_lora_a")
    return out


def moe_lora_route(handle: Handle, router_logits: torch.Tensor, top_k: int, routing_method: int = 0,
                   correction_bias: Optional[torch.Tensor] = None, routed_scaling_factor: float = 1.0,
                   n_group: int = 1, topk_group: int = 1, outputs: Optional[dict] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> dict:
    T, E = router_logits.shape
    dev = router_logits.device
    P = T * top_k
    o = dict(outputs or {})
    o.setdefault("topk_ids", torch.empty((T, top_k), dtype=torch.int32, device=dev))
    o.setdefault("topk_weights", torch.empty((T, top_k), dtype=torch.float32, device=dev))
    o.setdefault("expert_offsets", torch.empty((E + 1,), dtype=torch.int32, device=dev))
    o.setdefault("perm", torch.empty((P,), dtype=torch.int32, device=dev))
    o.setdefault("inv_perm", torch.empty((P,), dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = alloc_workspace(T, 0, 0, E, top_k, device=dev)
    st = lib().moe_lora_route(
        handle.ptr, _ptr(router_logits, torch.bfloat16, "router_logits"),
        _ptr(correction_bias, torch.float32, "correction_bias"), T, E, int(top_k), int(routing_method),
        float(routed_scaling_factor), int(n_group), int(topk_group),
        _ptr(o["topk_ids"], torch.int32), _ptr(o["topk_weights"], torch.float32),
        _ptr(o["expert_offsets"], torch.int32), _ptr(o["perm"], torch.int32), _ptr(o["inv_perm"], torch.int32),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "moe_lora_route")
    o["workspace"] = workspace
    return o


def moe_lora_permute(handle: Handle, hidden: torch.Tensor, perm: torch.Tensor, top_k: int,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    T, H = hidden.shape
    if out is None:
        out = torch.empty((T * top_k, H), dtype=torch.bfloat16, device=hidden.device)
    st = lib().moe_lora_permute(handle.ptr, _ptr(hidden, torch.bfloat16, "hidden"), _ptr(perm, torch.int32, "perm"),
                                T, H, int(top_k), _ptr(out, torch.bfloat16, "out"), _stream(stream))
    _check(st, "moe_lora_permute")
    return out


def check_shapes(hidden, router_logits, w1, w2, lora_A_gu=None, lora_B_gu=None, lora_A_dn=None,
                 lora_B_dn=None, slot_idx=None, ranks: Sequence[int] = (), scalings: Sequence[float] = (),
                 flags=0, num_experts=None, correction_bias=None, packed_k=False):
    """Raise ValueError unless every tensor has the shape the C ABI reads through its pointer:
    hidden [T, H], router_logits [T, E], w1 [E, 2I, H], w2 [E, H, I] (with packed_k, two values
    per byte along K: w1 [E, 2I, H/2], w2 [E, H, I/2]) and, with adapters,
    lora_A_gu [S, E', R, H], lora_B_gu [S, E, 2I, R], lora_A_dn [S, E, R, I],
    lora_B_dn [S, E', H, R] (E' = 1 with FLAG_SHARED_OUTER, else E) and slot_idx [T].
    The library takes raw pointers and cannot check these itself."""
    def need(t, shape, name):
        if t is None:
            raise ValueError(f"{name} is required")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if hidden.dim() != 2 or w1.dim() != 3:
        raise ValueError("hidden must be [T, H] and w1 [E, 2I, H]")
    T, H = hidden.shape
    E, twoI = w1.shape[0], w1.shape[1]
    if twoI % 2:
        raise ValueError(f"w1's second dimension (2I) must be even, got {twoI}")
    I = twoI // 2
    if packed_k:
        if H % 2:
            raise ValueError(f"H must be even, got {H}")
        need(w1, (E, twoI, H // 2), "w1")
        if w2.dim() != 3 or w2.shape[:2] != (E, H):
            raise ValueError(f"w2 must have shape ({E}, {H}, I/2), got {tuple(w2.shape)}")
        if w2.shape[2] * 2 != I:
            raise ValueError(f"w2's last dimension must be I/2 = {I // 2}, got {w2.shape[2]}")
    else:
        need(w1, (E, twoI, H), "w1")
        need(w2, (E, H, I), "w2")
    if router_logits is not None:
        need(router_logits, (T, num_experts if num_experts is not None else E), "router_logits")
    if correction_bias is not None:
        need(correction_bias, (router_logits.shape[1] if router_logits is not None else E,), "correction_bias")
    S = len(ranks)
    if len(scalings) != S:
        raise ValueError(f"ranks and scalings must have the same length, got {S} and {len(scalings)}")
    if S == 0:
        return
    if lora_A_gu is None or lora_A_gu.dim() != 4:
        raise ValueError("lora_A_gu [S, E, R, H] is required with adapters")
    R = lora_A_gu.shape[2]
    Eo = 1 if (int(flags) & FLAG_SHARED_OUTER) else E
    need(lora_A_gu, (S, Eo, R, H), "lora_A_gu")
    need(lora_B_gu, (S, E, twoI, R), "lora_B_gu")
    need(lora_A_dn, (S, E, R, I), "lora_A_dn")
    need(lora_B_dn, (S, Eo, H, R), "lora_B_dn")
    need(slot_idx, (T,), "slot_idx")
    if any(int(r) > R or int(r) < 0 for r in ranks):
        raise ValueError(f"every rank must lie in [0, R = {R}], got {list(ranks)}")


def make_args(hidden, router_logits, w1, w2, top_k, routing_method=0, correction_bias=None,
              routed_scaling_factor=1.0, lora_A_gu=None, lora_B_gu=None, lora_A_dn=None, lora_B_dn=None,
              slot_idx=None, ranks: Sequence[int] = (), scalings: Sequence[float] = (), flags=0,
              outputs: Optional[dict] = None, prof_events=None, n_group=1, topk_group=1,
              weight_dtype=torch.bfloat16, packed_k=False, lora_B_gu_packed=None, lora_B_dn_packed=None,
              lora_A_gu_packed=None, lora_A_dn_packed=None):
    """Fill the C argument struct.  Returns (Args, keepalive) -- keep both alive for the call."""
    check_shapes(hidden, router_logits, w1, w2, lora_A_gu, lora_B_gu, lora_A_dn, lora_B_dn, slot_idx, ranks,
                 scalings, flags, correction_bias=correction_bias, packed_k=packed_k)
    for t, name, Eb, N, gated in (
            (lora_B_gu_packed, "lora_B_gu_packed", w1.shape[0], w1.shape[1], 1),
            (lora_B_dn_packed, "lora_B_dn_packed", 1 if (int(flags) & FLAG_SHARED_OUTER) else w1.shape[0],
             hidden.shape[1], 0)):
        if t is not None:
            want = packed_lora_b_shape(Eb, N, gated, ranks)
            if tuple(t.shape) != want:
                raise ValueError(f"{name} must have shape {want} (moe_lora_pack_lora_b with these ranks), "
                                 f"got {tuple(t.shape)}")
    for t, name, Ea, K in (
            (lora_A_gu_packed, "lora_A_gu_packed", 1 if (int(flags) & FLAG_SHARED_OUTER) else w1.shape[0],
             hidden.shape[1]),
            (lora_A_dn_packed, "lora_A_dn_packed", w1.shape[0], w1.shape[1] // 2)):
        if t is not None:
            want = packed_lora_a_shape(Ea, K, ranks)
            if tuple(t.shape) != want:
                raise ValueError(f"{name} must have shape {want} (moe_lora_pack_lora_a with these ranks), "
                                 f"got {tuple(t.shape)}")
    T, H = hidden.shape
    E, twoI, _ = w1.shape
    S = len(ranks)
    R = int(lora_A_gu.shape[2]) if (lora_A_gu is not None and S > 0) else 0
    ranks_arr = (ctypes.c_int32 * max(S, 1))(*[int(r) for r in ranks])
    scal_arr = (c_float * max(S, 1))(*[float(s) for s in scalings])
    o = outputs or {}
    a = Args()
    a.T, a.H, a.I, a.E, a.top_k, a.S, a.R = T, H, twoI // 2, E, int(top_k), S, R
    a.routing_method, a.routed_scaling_factor = int(routing_method), float(routed_scaling_factor)
    a.n_group, a.topk_group = int(n_group), int(topk_group)
    a.hidden = _ptr(hidden, torch.bfloat16, "hidden")
    a.router_logits = _ptr(router_logits, torch.bfloat16, "router_logits")
    a.correction_bias = _ptr(correction_bias, torch.float32, "correction_bias")
    a.w1 = _ptr(w1, weight_dtype, "w1")
    a.w2 = _ptr(w2, weight_dtype, "w2")
    a.lora_A_gu = _ptr(lora_A_gu, torch.bfloat16, "lora_A_gu")
    a.lora_B_gu = _ptr(lora_B_gu, torch.bfloat16, "lora_B_gu")
    a.lora_A_dn = _ptr(lora_A_dn, torch.bfloat16, "lora_A_dn")
    a.lora_B_dn = _ptr(lora_B_dn, torch.bfloat16, "lora_B_dn")
    a.slot_idx = _ptr(slot_idx, torch.int32, "slot_idx")
    a.h_ranks = ranks_arr
    a.h_scalings = scal_arr
    a.flags = int(flags)
    a.topk_ids = _ptr(o.get("topk_ids"), torch.int32)
    a.topk_weights = _ptr(o.get("topk_weights"), torch.float32)
    a.expert_offsets = _ptr(o.get("expert_offsets"), torch.int32)
    a.perm = _ptr(o.get("perm"), torch.int32)
    a.inv_perm = _ptr(o.get("inv_perm"), torch.int32)
    a.lora_B_gu_packed = _ptr(lora_B_gu_packed, torch.bfloat16, "lora_B_gu_packed")
    a.lora_B_dn_packed = _ptr(lora_B_dn_packed, torch.bfloat16, "lora_B_dn_packed")
    a.lora_A_gu_packed = _ptr(lora_A_gu_packed, torch.bfloat16, "lora_A_gu_packed")
    a.lora_A_dn_packed = _ptr(lora_A_dn_packed, torch.bfloat16, "lora_A_dn_packed")
    ev_arr = None
    if prof_events is not None:
        ev_arr = (c_void_p * (2 * NUM_STAGES))(*[(e.cuda_event if e is not None else None) for e in prof_events])
        a.prof_events = ctypes.cast(ev_arr, c_void_p)
    return a, (ranks_arr, scal_arr, ev_arr)


def moe_lora_forward(handle: Handle, hidden, router_logits, w1, w2, top_k, routing_method=0,
                     correction_bias=None, routed_scaling_factor=1.0, lora_A_gu=None, lora_B_gu=None,
                     lora_A_dn=None, lora_B_dn=None, slot_idx=None, ranks=(), scalings=(), flags=0,
                     out=None, workspace=None, outputs=None, prof_events=None, stream=None,
                     n_group=1, topk_group=1, lora_B_gu_packed=None, lora_B_dn_packed=None,
                     lora_A_gu_packed=None, lora_A_dn_packed=None) -> torch.Tensor:
    """The whole layer: returns out [T, H] bf16 (written in place when `out` is given).
    lora_B_*_packed / lora_A_*_packed: optional expand-ready and shrink-ready copies
    (moe_lora_pack_lora_b / moe_lora_pack_lora_a) made with the same ranks."""
    a, keep = make_args(hidden, router_logits, w1, w2, top_k, routing_method, correction_bias,
                        routed_scaling_factor, lora_A_gu, lora_B_gu, lora_A_dn, lora_B_dn, slot_idx, ranks,
                        scalings, flags, outputs, prof_events, n_group, topk_group,
                        lora_B_gu_packed=lora_B_gu_packed, lora_B_dn_packed=lora_B_dn_packed,
                        lora_A_gu_packed=lora_A_gu_packed, lora_A_dn_packed=lora_A_dn_packed)
    if out is None:
        out = torch.empty((a.T, a.H), dtype=torch.bfloat16, device=hidden.device)
    if workspace is None:
        workspace = alloc_workspace(a.T, a.H, a.I, a.E, a.top_k, a.S, a.R, device=hidden.device)
    st = lib().moe_lora_forward(handle.ptr, ctypes.byref(a), _ptr(out, torch.bfloat16, "out"),
                                _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "moe_lora_forward")
    del keep
    return out


def moe_lora_forward_routed(handle: Handle, hidden, packed_topk_ids, w1, w2, top_k, num_experts,
                            local_expert_offset=0, do_finalize=True, lora_A_gu=None, lora_B_gu=None,
                            lora_A_dn=None, lora_B_dn=None, slot_idx=None, ranks=(), scalings=(), flags=0,
                            out=None, gemm2_output=None, activation_output=None, expert_weights=None,
                            expanded_idx_to_permuted_idx=None, workspace=None, stream=None):
    """The layer with the routing given as packed top-k words [T, top_k] int32
    ((global expert << 16) | bf16 weight bits); w1/w2/LoRA hold the local experts
    [local_expert_offset, local_expert_offset + E).  do_finalize=True returns out [T, H]
    bf16; False returns a dict of gemm2_output [T*k, H] fp32, activation_output [T*k, I]
    bf16, expert_weights [T, k] fp32 and expanded_idx_to_permuted_idx [T*k] int32 (-1 for
    pairs of non-local experts)."""
    T, H = hidden.shape
    E, twoI, _ = w1.shape
    dev = hidden.device
    a, keep = make_args(hidden, None, w1, w2, top_k, 0, None, 1.0, lora_A_gu, lora_B_gu, lora_A_dn, lora_B_dn,
                        slot_idx, ranks, scalings, flags)
    P = T * int(top_k)
    r = Routed()
    r.packed_topk_ids = _ptr(packed_topk_ids, torch.int32, "packed_topk_ids")
    r.num_experts, r.local_expert_offset, r.do_finalize = int(num_experts), int(local_expert_offset), int(bool(do_finalize))
    if expert_weights is None:
        expert_weights = torch.empty((T, top_k), dtype=torch.float32, device=dev)
    if expanded_idx_to_permuted_idx is None:
        expanded_idx_to_permuted_idx = torch.empty((P,), dtype=torch.int32, device=dev)
    r.expert_weights = _ptr(expert_weights, torch.float32, "expert_weights")
    r.expanded_idx_to_permuted_idx = _ptr(expanded_idx_to_permuted_idx, torch.int32, "expanded_idx_to_permuted_idx")
    if do_finalize:
        if out is None:
            out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    else:
        if gemm2_output is None:
            gemm2_output = torch.empty((P, H), dtype=torch.float32, device=dev)
        if activation_output is None:
            activation_output = torch.empty((P, twoI // 2), dtype=torch.bfloat16, device=dev)
        r.gemm2_output = _ptr(gemm2_output, torch.float32, "gemm2_output")
        r.activation_output = _ptr(activation_output, torch.bfloat16, "activation_output")
    if workspace is None:
        workspace = alloc_workspace(T, H, twoI // 2, E, top_k, a.S, a.R, device=dev)
    st = lib().moe_lora_forward_routed(handle.ptr, ctypes.byref(a), ctypes.byref(r),
                                       _ptr(out, torch.bfloat16, "out") if do_finalize else None,
                                       _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "moe_lora_forward_routed")
    del keep
    if do_finalize:
        return out
    return dict(gemm2_output=gemm2_output, activation_output=activation_output, expert_weights=expert_weights,
                expanded_idx_to_permuted_idx=expanded_idx_to_permuted_idx)


def check_fp8_weights(w1_q, w1_scale, w2_q, w2_scale):
    """Raise ValueError unless the FP8 weights have the shapes the C ABI reads: codes
    w1_q [E, 2I, H] and w2_q [E, H, I] (uint8), block scales w1_scale [E, 2I/128, H/128]
    and w2_scale [E, H/128, I/128] (float32), H and I multiples of 128."""
    if w1_q.dim() != 3 or w2_q.dim() != 3:
        raise ValueError("w1_q must be [E, 2I, H] and w2_q [E, H, I]")
    E, twoI, H = w1_q.shape
    I = twoI // 2
    if H % 128 or I % 128 or twoI % 2:
        raise ValueError(f"H and I must be multiples of 128, got H={H}, I={I}")
    for t, shape, name in ((w2_q, (E, H, I), "w2_q"), (w1_scale, (E, twoI // 128, H // 128), "w1_scale"),
                           (w2_scale, (E, H // 128, I // 128), "w2_scale")):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")


def moe_lora_forward_fp8(handle: Handle, hidden, router_logits, w1_q, w1_scale, w2_q, w2_scale, top_k,
                         routing_method=0, correction_bias=None, routed_scaling_factor=1.0, lora_A_gu=None,
                         lora_B_gu=None, lora_A_dn=None, lora_B_dn=None, slot_idx=None, ranks=(), scalings=(),
                         flags=0, out=None, workspace=None, outputs=None, prof_events=None, stream=None,
                         n_group=1, topk_group=1, lora_B_gu_packed=None, lora_B_dn_packed=None,
                         lora_A_gu_packed=None, lora_A_dn_packed=None) -> torch.Tensor:
    """The layer with FP8 block-scale expert weights: w1_q [E, 2I, H] and w2_q [E, H, I] hold
    e4m3 bit patterns (uint8), w1_scale [E, 2I/128, H/128] and w2_scale [E, H/128, I/128]
    the float32 scales of their 128 x 128 blocks.  With both expand-ready LoRA B copies
    (moe_lora_pack_lora_b) the fused LoRA placement runs.  Returns out [T, H] bf16."""
    check_fp8_weights(w1_q, w1_scale, w2_q, w2_scale)
    a, keep = make_args(hidden, router_logits, w1_q, w2_q, top_k, routing_method, correction_bias,
                        routed_scaling_factor, lora_A_gu, lora_B_gu, lora_A_dn, lora_B_dn, slot_idx, ranks,
                        scalings, flags, outputs, prof_events, n_group, topk_group, weight_dtype=torch.uint8,
                        lora_B_gu_packed=lora_B_gu_packed, lora_B_dn_packed=lora_B_dn_packed,
                        lora_A_gu_packed=lora_A_gu_packed, lora_A_dn_packed=lora_A_dn_packed)
    w = Fp8Weights()
    w.w1 = _ptr(w1_q, torch.uint8, "w1_q")
    w.w1_scale = _ptr(w1_scale, torch.float32, "w1_scale")
    w.w2 = _ptr(w2_q, torch.uint8, "w2_q")
    w.w2_scale = _ptr(w2_scale, torch.float32, "w2_scale")
    if out is None:
        out = torch.empty((a.T, a.H), dtype=torch.bfloat16, device=hidden.device)
    if workspace is None:
        workspace = alloc_workspace(a.T, a.H, a.I, a.E, a.top_k, a.S, a.R, device=hidden.device)
    st = lib().moe_lora_forward_fp8(handle.ptr, ctypes.byref(a), ctypes.byref(w), _ptr(out, torch.bfloat16, "out"),
                                    _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "moe_lora_forward_fp8")
    del keep
    return out


def moe_lora_quant_fp8(handle: Handle, src: torch.Tensor, perm: Optional[torch.Tensor] = None, top_k: int = 1,
                       stream=None):
    """FP8 group quantisation of bf16 rows src [T, K]: returns (codes [rows, K] uint8 e4m3
    bit patterns, scales [K/128, rows] float32).  With perm [T*top_k], output row q
    quantises src row perm[q] // top_k (rows = T*top_k); without it rows = T."""
    T, K = src.shape
    rows = perm.numel() if perm is not None else T
    codes = torch.empty((rows, K), dtype=torch.uint8, device=src.device)
    scales = torch.empty((K // 128, rows), dtype=torch.float32, device=src.device)
    st = lib().moe_lora_quant_fp8(handle.ptr, _ptr(src, torch.bfloat16, "src"), _ptr(perm, torch.int32, "perm"),
                                  rows, K, int(top_k), _ptr(codes, torch.uint8), _ptr(scales, torch.float32),
                                  _stream(stream))
    _check(st, "moe_lora_quant_fp8")
    return codes, scales


def moe_lora_grouped_gemm_fp8(handle: Handle, w_q: torch.Tensor, w_scale: torch.Tensor, x_q: torch.Tensor,
                              x_scale: torch.Tensor, expert_offsets: torch.Tensor, stream=None) -> torch.Tensor:
    """The FP8 block-scaled grouped GEMM on its own: w_q [E, N, K] and x_q [P, K] e4m3 codes
    (uint8), w_scale [E, N/128, K/128] and x_scale [K/128, P] float32, expert_offsets [E + 1]
    int32.  Returns out [P, N] float32 (rows outside every expert's range are left as zero)."""
    if w_q.dim() != 3 or x_q.dim() != 2:
        raise ValueError("w_q must be [E, N, K] and x_q [P, K]")
    E, N, K = w_q.shape
    P = x_q.shape[0]
    for t, shape, name in ((x_q, (P, K), "x_q"), (w_scale, (E, N // 128, K // 128), "w_scale"),
                           (x_scale, (K // 128, P), "x_scale"), (expert_offsets, (E + 1,), "expert_offsets")):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    out = torch.zeros((P, N), dtype=torch.float32, device=w_q.device)
    st = lib().moe_lora_grouped_gemm_fp8(handle.ptr, _ptr(w_q, torch.uint8, "w_q"), _ptr(w_scale, torch.float32, "w_scale"),
                                         _ptr(x_q, torch.uint8, "x_q"), _ptr(x_scale, torch.float32, "x_scale"),
                                         _ptr(expert_offsets, torch.int32, "expert_offsets"), E, N, K, P,
                                         _ptr(out, torch.float32, "out"), _stream(stream))
    _check(st, "moe_lora_grouped_gemm_fp8")
    return out


def check_nvfp4_weights(w1_q, w1_sf, w1_gs, w2_q, w2_sf, w2_gs):
    """Raise ValueError unless the NVFP4 weights have the shapes the C ABI reads: packed codes
    w1_q [E, 2I, H/2] and w2_q [E, H, I/2] (uint8), block scales w1_sf [E, 2I, H/16] and
    w2_sf [E, H, I/16] (uint8 e4m3 bit patterns), tensor scales w1_gs and w2_gs [E] (float32);
    H a multiple of 128, I of 64."""
    if w1_q.dim() != 3 or w2_q.dim() != 3:
        raise ValueError("w1_q must be [E, 2I, H/2] and w2_q [E, H, I/2]")
    E, twoI, H2 = w1_q.shape
    H, I = 2 * H2, twoI // 2
    if H % 128 or I % 64 or twoI % 2:
        raise ValueError(f"H must be a multiple of 128 and I of 64, got H={H}, I={I}")
    for t, shape, name in ((w2_q, (E, H, I // 2), "w2_q"), (w1_sf, (E, twoI, H // 16), "w1_sf"),
                           (w2_sf, (E, H, I // 16), "w2_sf"), (w1_gs, (E,), "w1_gs"), (w2_gs, (E,), "w2_gs")):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")


def moe_lora_forward_nvfp4(handle: Handle, hidden, router_logits, w1_q, w1_sf, w1_gs, w2_q, w2_sf, w2_gs, top_k,
                           routing_method=0, correction_bias=None, routed_scaling_factor=1.0, lora_A_gu=None,
                           lora_B_gu=None, lora_A_dn=None, lora_B_dn=None, slot_idx=None, ranks=(), scalings=(),
                           flags=0, out=None, workspace=None, outputs=None, prof_events=None, stream=None,
                           n_group=1, topk_group=1) -> torch.Tensor:
    """The layer with NVFP4 expert weights: packed e2m1 codes w1_q [E, 2I, H/2] and
    w2_q [E, H, I/2] (uint8, element 2i in the low nibble of byte i), e4m3 block scales
    w1_sf [E, 2I, H/16] and w2_sf [E, H, I/16] (uint8 bit patterns), float32 tensor scales
    w1_gs and w2_gs [E].  Returns out [T, H] bf16."""
    check_nvfp4_weights(w1_q, w1_sf, w1_gs, w2_q, w2_sf, w2_gs)
    a, keep = make_args(hidden, router_logits, w1_q, w2_q, top_k, routing_method, correction_bias,
                        routed_scaling_factor, lora_A_gu, lora_B_gu, lora_A_dn, lora_B_dn, slot_idx, ranks,
                        scalings, flags, outputs, prof_events, n_group, topk_group, weight_dtype=torch.uint8,
                        packed_k=True)
    w = Nvfp4Weights()
    w.w1 = _ptr(w1_q, torch.uint8, "w1_q")
    w.w1_sf = _ptr(w1_sf, torch.uint8, "w1_sf")
    w.w1_gs = _ptr(w1_gs, torch.float32, "w1_gs")
    w.w2 = _ptr(w2_q, torch.uint8, "w2_q")
    w.w2_sf = _ptr(w2_sf, torch.uint8, "w2_sf")
    w.w2_gs = _ptr(w2_gs, torch.float32, "w2_gs")
    if out is None:
        out = torch.empty((a.T, a.H), dtype=torch.bfloat16, device=hidden.device)
    if workspace is None:
        workspace = alloc_workspace(a.T, a.H, a.I, a.E, a.top_k, a.S, a.R, device=hidden.device)
    st = lib().moe_lora_forward_nvfp4(handle.ptr, ctypes.byref(a), ctypes.byref(w), _ptr(out, torch.bfloat16, "out"),
                                      _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "moe_lora_forward_nvfp4")
    del keep
    return out


def moe_lora_quant_nvfp4(handle: Handle, src: torch.Tensor, perm: Optional[torch.Tensor] = None, top_k: int = 1,
                         stream=None):
    """NVFP4 row quantisation of bf16 rows src [T, K]: returns (g [rows] float32 row scales,
    codes [rows, K/2] uint8 packed e2m1, block_scales [rows, K/16] uint8 e4m3 bit patterns,
    deq [rows, K] float16 = e2m1 * block scale, the values the GEMMs read).  With perm
    [T*top_k], output row q quantises src row perm[q] // top_k (rows = T*top_k); without it
    rows = T."""
    T, K = src.shape
    rows = perm.numel() if perm is not None else T
    dev = src.device
    g = torch.empty((rows,), dtype=torch.float32, device=dev)
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty((rows, K // 16), dtype=torch.uint8, device=dev)
    deq = torch.empty((rows, K), dtype=torch.float16, device=dev)
    st = lib().moe_lora_quant_nvfp4(handle.ptr, _ptr(src, torch.bfloat16, "src"), _ptr(perm, torch.int32, "perm"),
                                    rows, K, int(top_k), _ptr(g, torch.float32), _ptr(codes, torch.uint8),
                                    _ptr(sf, torch.uint8), _ptr(deq, torch.float16), _stream(stream))
    _check(st, "moe_lora_quant_nvfp4")
    return g, codes, sf, deq


def moe_lora_grouped_gemm_nvfp4(handle: Handle, w_q: torch.Tensor, w_sf: torch.Tensor, w_gs: torch.Tensor,
                                x: torch.Tensor, x_gs: torch.Tensor, expert_offsets: torch.Tensor,
                                stream=None) -> torch.Tensor:
    """The NVFP4 grouped GEMM on its own: packed codes w_q [E, N, K/2], block scales
    w_sf [E, N, K/16] (uint8), tensor scales w_gs [E] and row scales x_gs [P] (float32),
    inputs x [P, K] float16 (the exact values of moe_lora_quant_nvfp4), expert_offsets [E + 1]
    int32.  Returns out [P, N] float32 (rows outside every expert's range are left as zero)."""
    if w_q.dim() != 3 or x.dim() != 2:
        raise ValueError("w_q must be [E, N, K/2] and x [P, K]")
    E, N, K2 = w_q.shape
    K = 2 * K2
    P = x.shape[0]
    for t, shape, name in ((x, (P, K), "x"), (w_sf, (E, N, K // 16), "w_sf"), (w_gs, (E,), "w_gs"),
                           (x_gs, (P,), "x_gs"), (expert_offsets, (E + 1,), "expert_offsets")):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    out = torch.zeros((P, N), dtype=torch.float32, device=w_q.device)
    st = lib().moe_lora_grouped_gemm_nvfp4(handle.ptr, _ptr(w_q, torch.uint8, "w_q"), _ptr(w_sf, torch.uint8, "w_sf"),
                                           _ptr(w_gs, torch.float32, "w_gs"), _ptr(x, torch.float16, "x"),
                                           _ptr(x_gs, torch.float32, "x_gs"),
                                           _ptr(expert_offsets, torch.int32, "expert_offsets"), E, N, K, P,
                                           _ptr(out, torch.float32, "out"), _stream(stream))
    _check(st, "moe_lora_grouped_gemm_nvfp4")
    return out


def moe_lora_validate(**kwargs) -> int:
    a, keep = make_args(**kwargs)
    return lib().moe_lora_validate(ctypes.byref(a))


def moe_lora_check_status(workspace: torch.Tensor, stream=None):
    """Synchronize `stream` and return (status, raw_word) of the last call on `workspace`."""
    word = ctypes.c_uint32()
    st = lib().moe_lora_check_status(_ptr(workspace, torch.uint8, "workspace"), _stream(stream), ctypes.byref(word))
    return st, word.value
