"""Python binding of the GB300 MoE layer library (libmoe.so, C ABI in include/moe.h).

Argument marshalling only: every function takes torch CUDA tensors, checks them, and calls
the C entry point of the same name on the current CUDA stream.  There is no fallback: if
libmoe.so is missing or fails to load, importing the compute functions raises.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_INDEX, ERR_TIMEOUT, ERR_DEVICE_CHECK = range(8)
SCORE_SOFTMAX, SCORE_SQRT_SOFTPLUS = 0, 1
W_MXFP4, W_NVFP4, W_INT8, W_INT8_B256 = 0, 1, 2, 3
SCORE_FNS = {"softmax": SCORE_SOFTMAX, "sqrt_softplus": SCORE_SQRT_SOFTPLUS}
WFMTS = {"mxfp4": W_MXFP4, "nvfp4": W_NVFP4, "int8": W_INT8, "int8b": W_INT8_B256}
I8_FMTS = (W_INT8, W_INT8_B256)


class MoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


class _Weight(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("tscale", ctypes.c_void_p), ("fmt", ctypes.c_int),
                ("E", ctypes.c_int), ("N", ctypes.c_int), ("Kd", ctypes.c_int), ("pair", ctypes.c_int)]


_lib = None


def lib():
    """The loaded libmoe.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not found: build it with `python -m moe_expert_ffn_sqrt_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int
        L.moe_msum_upper.restype = Z
        L.moe_msum_upper.argtypes = [I, I, I, I]
        L.moe_act_sf_block_rows.restype = I
        L.moe_act_sf_block_rows.argtypes = [I]
        L.moe_act_sf_tiled_bytes.restype = Z
        L.moe_act_sf_tiled_bytes.argtypes = [I, I, I]
        L.moe_act_sf_untile_host.restype = S
        L.moe_act_sf_untile_host.argtypes = [P, I, I, I, P]
        L.moe_act_sf_tile_host.restype = S
        L.moe_act_sf_tile_host.argtypes = [P, I, I, I, P]
        L.moe_weight_packed_bytes.restype = Z
        L.moe_weight_packed_bytes.argtypes = [I, I, I, I, I]
        L.moe_pack_weights.restype = S
        L.moe_pack_weights.argtypes = [I, P, P, I, I, I, I, P, P]
        L.moe_workspace_size.restype = S
        L.moe_workspace_size.argtypes = [I, I, I, I, I, I, ctypes.POINTER(Z)]
        L.moe_route.restype = S
        L.moe_route.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, Z, P]
        L.moe_route_noalloc.restype = S
        L.moe_route_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P]
        L.moe_permute.restype = S
        L.moe_permute.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, I, P, P, P, Z, P]
        L.moe_grouped_gemm_l1_swiglu.restype = S
        L.moe_grouped_gemm_l1_swiglu.argtypes = [P, P, I, P, P, P, I, I, I, I, I, I, _Weight, P, P, P, Z, P]
        L.moe_grouped_gemm_l2.restype = S
        L.moe_grouped_gemm_l2.argtypes = [P, P, P, P, I, I, I, I, I, I, _Weight, P, P, Z, P]
        L.moe_grouped_ffn.restype = S
        L.moe_grouped_ffn.argtypes = [P, P, I, P, P, P, I, I, I, I, I, I, _Weight, _Weight, P, P, P, P, Z, P]
        L.moe_unpermute_reduce.restype = S
        L.moe_unpermute_reduce.argtypes = [P, P, P, I, I, I, P, P]
        L.moe_forward.restype = S
        L.moe_forward.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, _Weight, _Weight, P, P, P, P, P, P, P, P, Z, P]
        L.moe_batched_align.restype = I
        L.moe_batched_align.argtypes = [I, I, I, I]
        L.moe_workspace_size_batched.restype = S
        L.moe_workspace_size_batched.argtypes = [I, I, I, I, I, I, ctypes.POINTER(Z)]
        L.moe_permute_batched.restype = S
        L.moe_permute_batched.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, I, P, P, P, Z, P]
        L.moe_grouped_ffn_batched.restype = S
        L.moe_grouped_ffn_batched.argtypes = [P, P, P, I, I, I, I, I, I, _Weight, _Weight, P, P, P, P, Z, P]
        L.moe_forward_batched.restype = S
        L.moe_forward_batched.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, _Weight, _Weight, P, P, P, P, P, P, P,
                                          P, P, Z, P]
        L.moe_grouped_gemm_l1_swiglu_weighted.restype = S
        L.moe_grouped_gemm_l1_swiglu_weighted.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, _Weight, P, P, P, Z, P]
        L.moe_forward_l1_weighted.restype = S
        L.moe_forward_l1_weighted.argtypes = L.moe_forward.argtypes
        L.moe_forward_single_launch.restype = S
        L.moe_forward_single_launch.argtypes = L.moe_forward.argtypes
        L.moe_route_naive.restype = S
        L.moe_route_naive.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, Z, P]
        L.moe_forward_naive.restype = S
        L.moe_forward_naive.argtypes = [P, P, P, P, I, I, I, I, I, I, I, _Weight, _Weight, P, P, P, P, P, P, P, P,
                                        Z, P]
        L.moe_selftest_wait_timeout.restype = S
        L.moe_workspace_size_i8.argtypes = [I, I, I, I, I, I, ctypes.POINTER(Z)]
        L.moe_workspace_size_i8.restype = S
        L.moe_act_quant_i8.argtypes = [P, I, I, P, P, P]
        L.moe_act_quant_i8.restype = S
        L.moe_act_quant_i8_b256.argtypes = [P, I, I, P, P, P]
        L.moe_act_quant_i8_b256.restype = S
        L.moe_grouped_gemm_l1_swiglu_i8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, _Weight, P, P, P, Z, P]
        L.moe_grouped_gemm_l1_swiglu_i8.restype = S
        L.moe_grouped_gemm_l2_i8.argtypes = [P, P, P, P, I, I, I, I, I, I, _Weight, P, P, Z, P]
        L.moe_grouped_gemm_l2_i8.restype = S
        L.moe_forward_i8.argtypes = L.moe_forward.argtypes
        L.moe_forward_i8.restype = S
        L.moe_workspace_size_batched_i8.argtypes = [I, I, I, I, I, I, ctypes.POINTER(Z)]
        L.moe_workspace_size_batched_i8.restype = S
        L.moe_forward_batched_i8.argtypes = L.moe_forward_batched.argtypes
        L.moe_forward_batched_i8.restype = S
        L.moe_selftest_wait_timeout.argtypes = [P, Z, I, P]
        L.moe_get_error.restype = S
        L.moe_get_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int)]
        L.moe_status_str.restype = ctypes.c_char_p
        L.moe_status_str.argtypes = [I]
        _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().moe_status_str(int(s)).decode()


def _check(status, where):
    if status != OK:
        raise MoeError(status, where)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


# ---------------------------------------------------------------------------------- sizes

def msum_upper(T, K, E, align):
    return int(lib().moe_msum_upper(T, K, E, align))


def act_sf_block_rows(align):
    return int(lib().moe_act_sf_block_rows(align))


def act_sf_tiled_bytes(rows, slabs, align):
    return int(lib().moe_act_sf_tiled_bytes(rows, slabs, align))


def act_sf_untile(tiled, rows, slabs, align):
    """Host helper: tiled activation scales (numpy uint8) -> numpy [rows, slabs]."""
    import numpy as np
    src = np.ascontiguousarray(np.asarray(tiled, dtype=np.uint8).reshape(-1))
    if src.size < act_sf_tiled_bytes(rows, slabs, align):
        raise ValueError("tiled buffer too small")
    out = np.empty((rows, slabs), dtype=np.uint8)
    _check(lib().moe_act_sf_untile_host(src.ctypes.data, rows, slabs, align, out.ctypes.data),
           "moe_act_sf_untile_host")
    return out


def act_sf_tile(plain, align):
    """Host helper: numpy [rows, slabs] activation scales -> numpy tiled layout (1-D uint8)."""
    import numpy as np
    src = np.ascontiguousarray(np.asarray(plain, dtype=np.uint8))
    rows, slabs = src.shape
    out = np.empty(act_sf_tiled_bytes(rows, slabs, align), dtype=np.uint8)
    _check(lib().moe_act_sf_tile_host(src.ctypes.data, rows, slabs, align, out.ctypes.data), "moe_act_sf_tile_host")
    return out


def weight_packed_bytes(fmt, E, N, Kd, pair):
    return int(lib().moe_weight_packed_bytes(WFMTS.get(fmt, fmt), E, N, Kd, pair))


def workspace_size(T, H, I, E, K, align):
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(T, H, I, E, K, align, ctypes.byref(n)), "moe_workspace_size")
    return int(n.value)


def new_workspace(T, H, I, E, K, align, device="cuda"):
    """A zero-filled workspace tensor of the size moe_workspace_size() asks for."""
    return torch.zeros(workspace_size(T, H, I, E, K, align), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------------- weights

def pack_weights(fmt, q, sf, pair, out=None):
    """Packs codes q and scales sf into the GEMMs' weight stream (moe_pack_weights).

    FP4 formats: q [E, N, Kd/2] packed E2M1 (uint8), sf the block scales.  INT8 ("int8", "int8b"):
    q [E, N, Kd] int8, sf unused (the channel or block scales are passed to Weight as tscale).
    """
    if WFMTS.get(fmt, fmt) in I8_FMTS:
        E, N, Kd = q.shape
        qp, sfp = _ptr(q, torch.int8, "q"), None
    else:
        E, N, half = q.shape
        Kd = 2 * half
        qp, sfp = _ptr(q, torch.uint8, "q"), _ptr(sf, torch.uint8, "sf")
    if out is None:
        out = torch.empty(weight_packed_bytes(fmt, E, N, Kd, pair), dtype=torch.uint8, device=q.device)
    _check(lib().moe_pack_weights(WFMTS.get(fmt, fmt), qp, sfp, E, N, Kd, pair, _ptr(out, torch.uint8, "out"),
                                  _stream()), "moe_pack_weights")
    return out


class Weight:
    """One stacked expert weight tensor [E, N, Kd] on the device, packed for the grouped GEMMs.

    pair = 2 for W13 (gate rows 0..I-1 and up rows I..2I-1), 1 for W2.  The logical tensors are
    only read while packing.
    """

    def __init__(self, q, sf, tscale=None, fmt="mxfp4", pair=1):
        self.fmt = fmt
        self.E, self.N, kq = q.shape
        # INT8: tscale = [E, N] channel scales ("int8") or [E, N/256, Kd/256] block scales ("int8b")
        self.Kd = kq if WFMTS.get(fmt, fmt) in I8_FMTS else 2 * kq
        self.pair = pair
        self.tscale = tscale
        self.packed = pack_weights(fmt, q, sf, pair)

    def c(self):
        return _Weight(_ptr(self.packed, torch.uint8, "w.packed"), _ptr(self.tscale, torch.float32, "w.tscale"),
                       WFMTS.get(self.fmt, self.fmt), self.E, self.N, self.Kd, self.pair)


# ---------------------------------------------------------------------------------- hot path

def route(hidden, w_gate, gate_bias, e_score_bias, K, score_fn, renormalize, topk_ids, topk_w, ws,
          logits_out=None, x_q=None, x_sf=None):
    T, H = hidden.shape
    E = w_gate.shape[0]
    _check(lib().moe_route(_ptr(hidden, torch.bfloat16, "hidden"),
                           _ptr(w_gate, torch.float32, "w_gate"), _ptr(gate_bias, torch.float32, "gate_bias"),
                           _ptr(e_score_bias, torch.float32, "e_score_bias"), T, H, E, K,
                           SCORE_FNS.get(score_fn, score_fn), int(renormalize),
                           _ptr(logits_out, torch.float32, "logits_out"), _ptr(topk_ids, torch.int32, "topk_ids"),
                           _ptr(topk_w, torch.float32, "topk_w"), _ptr(x_q, torch.uint8, "x_q"),
                           _ptr(x_sf, torch.uint8, "x_sf"), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()),
           "moe_route")


def route_noalloc(hidden, w_gate, gate_bias, e_score_bias, K, score_fn, renormalize, topk_ids, topk_w,
                  logits_out=None, x_q=None, x_sf=None):
    """moe_route without a workspace (scratch lives in a fixed device array inside the library)."""
    T, H = hidden.shape
    E = w_gate.shape[0]
    _check(lib().moe_route_noalloc(_ptr(hidden, torch.bfloat16, "hidden"), _ptr(w_gate, torch.float32, "w_gate"),
                                   _ptr(gate_bias, torch.float32, "gate_bias"),
                                   _ptr(e_score_bias, torch.float32, "e_score_bias"), T, H, E, K,
                                   SCORE_FNS.get(score_fn, score_fn), int(renormalize),
                                   _ptr(logits_out, torch.float32, "logits_out"), _ptr(topk_ids, torch.int32, "topk_ids"),
                                   _ptr(topk_w, torch.float32, "topk_w"), _ptr(x_q, torch.uint8, "x_q"),
                                   _ptr(x_sf, torch.uint8, "x_sf"), _stream()), "moe_route_noalloc")


def permute(topk_ids, E, align, sorted_token_ids, expert_ids, inv_perm, m_sum, ws, expert_counts=None,
            x_q=None, x_sf=None, x_perm=None, x_perm_sf=None):
    """x_q/x_sf/x_perm/x_perm_sf: rows and scales copied; x_sf/x_perm_sf alone: the scales only."""
    T, K = topk_ids.shape
    H = x_q.shape[1] if x_q is not None else (x_sf.shape[1] * 128 if x_sf is not None else 0)
    _check(lib().moe_permute(_ptr(topk_ids, torch.int32, "topk_ids"), T, K, E, align,
                             _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                             _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(inv_perm, torch.int32, "inv_perm"),
                             _ptr(m_sum, torch.int32, "m_sum"), _ptr(expert_counts, torch.int32, "expert_counts"),
                             _ptr(x_q, torch.uint8, "x_q"), _ptr(x_sf, torch.uint8, "x_sf"), H,
                             _ptr(x_perm, torch.uint8, "x_perm"), _ptr(x_perm_sf, torch.uint8, "x_perm_sf"),
                             _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_permute")


def grouped_gemm_l1_swiglu(a_q, a_sf, expert_ids, m_sum, T, K, H, I, E, align, w13, h_q, h_sf, ws,
                           sorted_token_ids=None):
    """sorted_token_ids None: a_q / a_sf are the permuted rows x_perm [U, H] with tiled scales.  Given:
    a_q / a_sf are the token-order x_q [T, H] and x_sf [T, H/128], gathered through sorted_token_ids."""
    _check(lib().moe_grouped_gemm_l1_swiglu(_ptr(a_q, torch.uint8, "a_q"), _ptr(a_sf, torch.uint8, "a_sf"),
                                            int(sorted_token_ids is None),
                                            _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                                            _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(m_sum, torch.int32, "m_sum"),
                                            T, K, H, I, E, align, w13.c(), _ptr(h_q, torch.uint8, "h_q"),
                                            _ptr(h_sf, torch.uint8, "h_sf"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                            _stream()), "moe_grouped_gemm_l1_swiglu")


def grouped_gemm_l1_swiglu_weighted(x_perm, x_perm_sf, expert_ids, m_sum, sorted_token_ids, topk_w, T, K, H, I, E,
                                    align, w13, h_q, h_sf, ws):
    """L1 with the routing weight of each row's pair applied before the requant."""
    _check(lib().moe_grouped_gemm_l1_swiglu_weighted(
        _ptr(x_perm, torch.uint8, "x_perm"), _ptr(x_perm_sf, torch.uint8, "x_perm_sf"),
        _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(m_sum, torch.int32, "m_sum"),
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(topk_w, torch.float32, "topk_w"),
        T, K, H, I, E, align, w13.c(), _ptr(h_q, torch.uint8, "h_q"), _ptr(h_sf, torch.uint8, "h_sf"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_grouped_gemm_l1_swiglu_weighted")


def grouped_gemm_l2(h_q, h_sf, expert_ids, m_sum, T, K, H, I, E, align, w2, y_perm, ws):
    _check(lib().moe_grouped_gemm_l2(_ptr(h_q, torch.uint8, "h_q"), _ptr(h_sf, torch.uint8, "h_sf"),
                                     _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(m_sum, torch.int32, "m_sum"),
                                     T, K, H, I, E, align, w2.c(), _ptr(y_perm, torch.bfloat16, "y_perm"),
                                     _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_grouped_gemm_l2")


def grouped_ffn(a_q, a_sf, expert_ids, m_sum, T, K, H, I, E, align, w13, w2, h_q, h_sf, y_perm, ws,
                sorted_token_ids=None):
    """L1 + SwiGLU + requant and L2 in one call (one launch for MXFP4 weights); the L1 input as in
    grouped_gemm_l1_swiglu (permuted rows, or token-order rows gathered through sorted_token_ids)."""
    _check(lib().moe_grouped_ffn(_ptr(a_q, torch.uint8, "a_q"), _ptr(a_sf, torch.uint8, "a_sf"),
                                 int(sorted_token_ids is None), _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                                 _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(m_sum, torch.int32, "m_sum"),
                                 T, K, H, I, E, align, w13.c(), w2.c(), _ptr(h_q, torch.uint8, "h_q"),
                                 _ptr(h_sf, torch.uint8, "h_sf"), _ptr(y_perm, torch.bfloat16, "y_perm"),
                                 _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_grouped_ffn")


def unpermute_reduce(y_perm, inv_perm, topk_w, out):
    """topk_w None: plain sum (weights applied in L1)."""
    T, K = inv_perm.shape
    H = out.shape[1]
    _check(lib().moe_unpermute_reduce(_ptr(y_perm, torch.bfloat16, "y_perm"), _ptr(inv_perm, torch.int32, "inv_perm"),
                                      _ptr(topk_w, torch.float32, "topk_w"), T, K, H, _ptr(out, torch.bfloat16, "out"),
                                      _stream()), "moe_unpermute_reduce")


def forward(hidden, w_gate, gate_bias, e_score_bias, I, K, align, score_fn, renormalize, w13, w2, out, ws,
            topk_ids=None, topk_w=None, sorted_token_ids=None, expert_ids=None, inv_perm=None, m_sum=None,
            weights_in_l1=False, single_launch=False):
    """moe_forward; moe_forward_l1_weighted when weights_in_l1 (routing weights applied in L1);
    moe_forward_single_launch when single_launch (the whole layer in one launch, small batches)."""
    T, H = hidden.shape
    E = w_gate.shape[0]
    if weights_in_l1 and single_launch:
        raise MoeError(ERR_INVALID_ARG, "forward")
    fn = (lib().moe_forward_l1_weighted if weights_in_l1 else
          lib().moe_forward_single_launch if single_launch else lib().moe_forward)
    _check(fn(_ptr(hidden, torch.bfloat16, "hidden"), _ptr(w_gate, torch.float32, "w_gate"),
                             _ptr(gate_bias, torch.float32, "gate_bias"), _ptr(e_score_bias, torch.float32, "e_score_bias"),
                             T, H, I, E, K, align, SCORE_FNS.get(score_fn, score_fn), int(renormalize), w13.c(), w2.c(),
                             _ptr(out, torch.bfloat16, "out"), _ptr(topk_ids, torch.int32, "topk_ids"),
                             _ptr(topk_w, torch.float32, "topk_w"), _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                             _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(inv_perm, torch.int32, "inv_perm"),
                             _ptr(m_sum, torch.int32, "m_sum"), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()),
           "moe_forward_single_launch" if single_launch else "moe_forward")


# ------------------------------------------------------------------ BatchedExperts layout

def workspace_size_batched(T, H, I, E, K, max_tokens):
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size_batched(T, H, I, E, K, max_tokens, ctypes.byref(n)), "moe_workspace_size_batched")
    return int(n.value)


def new_workspace_batched(T, H, I, E, K, max_tokens, device="cuda"):
    """A zero-filled workspace tensor of the size moe_workspace_size_batched() asks for."""
    return torch.zeros(workspace_size_batched(T, H, I, E, K, max_tokens), dtype=torch.uint8, device=device)


def batched_align(T, K, E, max_tokens):
    """Row-block height (the `align`) of the BatchedExperts buffers' scale tiling and GEMMs."""
    a = int(lib().moe_batched_align(T, K, E, max_tokens))
    if a <= 0:
        raise MoeError(ERR_INVALID_ARG, "moe_batched_align")
    return a


def permute_batched(topk_ids, E, max_tokens, sorted_token_ids, expert_ids, inv_perm, m_sum, ws,
                    expert_num_tokens=None, x_q=None, x_sf=None, x_perm=None, x_perm_sf=None):
    T, K = topk_ids.shape
    H = x_q.shape[1] if x_q is not None else 0
    _check(lib().moe_permute_batched(_ptr(topk_ids, torch.int32, "topk_ids"), T, K, E, max_tokens,
                                     _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                                     _ptr(expert_ids, torch.int32, "expert_ids"),
                                     _ptr(inv_perm, torch.int32, "inv_perm"), _ptr(m_sum, torch.int32, "m_sum"),
                                     _ptr(expert_num_tokens, torch.int32, "expert_num_tokens"),
                                     _ptr(x_q, torch.uint8, "x_q"), _ptr(x_sf, torch.uint8, "x_sf"), H,
                                     _ptr(x_perm, torch.uint8, "x_perm"), _ptr(x_perm_sf, torch.uint8, "x_perm_sf"),
                                     _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_permute_batched")


def grouped_ffn_batched(x_perm, x_perm_sf, expert_num_tokens, T, K, H, I, E, max_tokens, w13, w2, h_q, h_sf, y_perm,
                        ws):
    """L1 + SwiGLU + requant and L2 over a BatchedExperts buffer [E * max_tokens, H]."""
    _check(lib().moe_grouped_ffn_batched(_ptr(x_perm, torch.uint8, "x_perm"), _ptr(x_perm_sf, torch.uint8, "x_perm_sf"),
                                         _ptr(expert_num_tokens, torch.int32, "expert_num_tokens"), T, K, H, I, E,
                                         max_tokens, w13.c(), w2.c(), _ptr(h_q, torch.uint8, "h_q"),
                                         _ptr(h_sf, torch.uint8, "h_sf"), _ptr(y_perm, torch.bfloat16, "y_perm"),
                                         _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_grouped_ffn_batched")


def forward_batched(hidden, w_gate, gate_bias, e_score_bias, I, K, max_tokens, score_fn, renormalize, w13, w2, out,
                    ws, topk_ids=None, topk_w=None, sorted_token_ids=None, expert_ids=None, inv_perm=None,
                    m_sum=None, expert_num_tokens=None):
    T, H = hidden.shape
    E = w_gate.shape[0]
    _check(lib().moe_forward_batched(
        _ptr(hidden, torch.bfloat16, "hidden"), _ptr(w_gate, torch.float32, "w_gate"),
        _ptr(gate_bias, torch.float32, "gate_bias"), _ptr(e_score_bias, torch.float32, "e_score_bias"),
        T, H, I, E, K, max_tokens, SCORE_FNS.get(score_fn, score_fn), int(renormalize), w13.c(), w2.c(),
        _ptr(out, torch.bfloat16, "out"), _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(topk_w, torch.float32, "topk_w"),
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(inv_perm, torch.int32, "inv_perm"), _ptr(m_sum, torch.int32, "m_sum"),
        _ptr(expert_num_tokens, torch.int32, "expert_num_tokens"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream()), "moe_forward_batched")


# ------------------------------------------------------------------ tiny-batch layout

NAIVE_ROWS = 16      # rows per (token, expert) pair; the GEMMs run with align = NAIVE_ROWS


def route_naive(hidden, w_gate, gate_bias, e_score_bias, K, score_fn, renormalize, topk_ids, topk_w,
                sorted_token_ids, expert_ids, inv_perm, m_sum, x_perm, x_perm_sf, ws):
    """Routing plus the tiny-batch layout (pair p on row 16p of the permuted buffers)."""
    T, H = hidden.shape
    E = w_gate.shape[0]
    _check(lib().moe_route_naive(
        _ptr(hidden, torch.bfloat16, "hidden"), _ptr(w_gate, torch.float32, "w_gate"),
        _ptr(gate_bias, torch.float32, "gate_bias"), _ptr(e_score_bias, torch.float32, "e_score_bias"), T, H, E, K,
        SCORE_FNS.get(score_fn, score_fn), int(renormalize), _ptr(topk_ids, torch.int32, "topk_ids"),
        _ptr(topk_w, torch.float32, "topk_w"), _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
        _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(inv_perm, torch.int32, "inv_perm"),
        _ptr(m_sum, torch.int32, "m_sum"), _ptr(x_perm, torch.uint8, "x_perm"), _ptr(x_perm_sf, torch.uint8, "x_perm_sf"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_route_naive")


def forward_naive(hidden, w_gate, gate_bias, e_score_bias, I, K, score_fn, renormalize, w13, w2, out, ws,
                  topk_ids=None, topk_w=None, sorted_token_ids=None, expert_ids=None, inv_perm=None, m_sum=None):
    """moe_forward over the tiny-batch layout (T <= 16, T*K <= E); ws sized for align 16."""
    T, H = hidden.shape
    E = w_gate.shape[0]
    _check(lib().moe_forward_naive(
        _ptr(hidden, torch.bfloat16, "hidden"), _ptr(w_gate, torch.float32, "w_gate"),
        _ptr(gate_bias, torch.float32, "gate_bias"), _ptr(e_score_bias, torch.float32, "e_score_bias"),
        T, H, I, E, K, SCORE_FNS.get(score_fn, score_fn), int(renormalize), w13.c(), w2.c(),
        _ptr(out, torch.bfloat16, "out"), _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(topk_w, torch.float32, "topk_w"),
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(inv_perm, torch.int32, "inv_perm"), _ptr(m_sum, torch.int32, "m_sum"), _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _stream()), "moe_forward_naive")


# ------------------------------------------------------------------ INT8 (W8A8) variant

def workspace_size_i8(T, H, I, E, K, align):
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size_i8(T, H, I, E, K, align, ctypes.byref(n)), "moe_workspace_size_i8")
    return int(n.value)


def new_workspace_i8(T, H, I, E, K, align, device="cuda"):
    """A zero-filled workspace tensor of the size moe_workspace_size_i8() asks for."""
    return torch.zeros(workspace_size_i8(T, H, I, E, K, align), dtype=torch.uint8, device=device)


def act_quant_i8(x, x_q, x_s):
    """Per-row int8 quantisation: x [R, C] bf16 -> x_q [R, C] int8, x_s [R] fp32; with x_s of shape
    [R, C/256], per 256-column group (moe_act_quant_i8_b256)."""
    R, C = x.shape
    fn = lib().moe_act_quant_i8_b256 if x_s.dim() == 2 else lib().moe_act_quant_i8
    _check(fn(_ptr(x, torch.bfloat16, "x"), R, C, _ptr(x_q, torch.int8, "x_q"), _ptr(x_s, torch.float32, "x_s"),
              _stream()), "moe_act_quant_i8")


def grouped_gemm_l1_swiglu_i8(x_q, x_s, sorted_token_ids, expert_ids, m_sum, T, K, H, I, E, align, w13, h_q, h_s, ws):
    """INT8 L1 + SwiGLU + per-row requant; x_q [T, H] in token order, gathered by sorted_token_ids."""
    _check(lib().moe_grouped_gemm_l1_swiglu_i8(
        _ptr(x_q, torch.int8, "x_q"), _ptr(x_s, torch.float32, "x_s"),
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(m_sum, torch.int32, "m_sum"), T, K, H, I, E, align, w13.c(), _ptr(h_q, torch.int8, "h_q"),
        _ptr(h_s, torch.float32, "h_s"), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()),
        "moe_grouped_gemm_l1_swiglu_i8")


def grouped_gemm_l2_i8(h_q, h_s, expert_ids, m_sum, T, K, H, I, E, align, w2, y_perm, ws):
    _check(lib().moe_grouped_gemm_l2_i8(_ptr(h_q, torch.int8, "h_q"), _ptr(h_s, torch.float32, "h_s"),
                                        _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(m_sum, torch.int32, "m_sum"),
                                        T, K, H, I, E, align, w2.c(), _ptr(y_perm, torch.bfloat16, "y_perm"),
                                        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()), "moe_grouped_gemm_l2_i8")


def forward_i8(hidden, w_gate, gate_bias, e_score_bias, I, K, align, score_fn, renormalize, w13, w2, out, ws,
               topk_ids=None, topk_w=None, sorted_token_ids=None, expert_ids=None, inv_perm=None, m_sum=None):
    """moe_forward_i8: the layer with INT8 weights and per-token INT8 activations."""
    T, H = hidden.shape
    E = w_gate.shape[0]
    _check(lib().moe_forward_i8(_ptr(hidden, torch.bfloat16, "hidden"), _ptr(w_gate, torch.float32, "w_gate"),
                                _ptr(gate_bias, torch.float32, "gate_bias"),
                                _ptr(e_score_bias, torch.float32, "e_score_bias"), T, H, I, E, K, align,
                                SCORE_FNS.get(score_fn, score_fn), int(renormalize), w13.c(), w2.c(),
                                _ptr(out, torch.bfloat16, "out"), _ptr(topk_ids, torch.int32, "topk_ids"),
                                _ptr(topk_w, torch.float32, "topk_w"),
                                _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                                _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(inv_perm, torch.int32, "inv_perm"),
                                _ptr(m_sum, torch.int32, "m_sum"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                _stream()), "moe_forward_i8")


def workspace_size_batched_i8(T, H, I, E, K, max_tokens):
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size_batched_i8(T, H, I, E, K, max_tokens, ctypes.byref(n)),
           "moe_workspace_size_batched_i8")
    return int(n.value)


def new_workspace_batched_i8(T, H, I, E, K, max_tokens, device="cuda"):
    """A zero-filled workspace tensor of the size moe_workspace_size_batched_i8() asks for."""
    return torch.zeros(workspace_size_batched_i8(T, H, I, E, K, max_tokens), dtype=torch.uint8, device=device)


def forward_batched_i8(hidden, w_gate, gate_bias, e_score_bias, I, K, max_tokens, score_fn, renormalize, w13, w2, out,
                       ws, topk_ids=None, topk_w=None, sorted_token_ids=None, expert_ids=None, inv_perm=None,
                       m_sum=None, expert_num_tokens=None):
    """moe_forward_batched_i8: the INT8 layer over the BatchedExperts layout."""
    T, H = hidden.shape
    E = w_gate.shape[0]
    _check(lib().moe_forward_batched_i8(
        _ptr(hidden, torch.bfloat16, "hidden"), _ptr(w_gate, torch.float32, "w_gate"),
        _ptr(gate_bias, torch.float32, "gate_bias"), _ptr(e_score_bias, torch.float32, "e_score_bias"), T, H, I, E, K,
        max_tokens, SCORE_FNS.get(score_fn, score_fn), int(renormalize), w13.c(), w2.c(),
        _ptr(out, torch.bfloat16, "out"), _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(topk_w, torch.float32, "topk_w"),
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(inv_perm, torch.int32, "inv_perm"), _ptr(m_sum, torch.int32, "m_sum"),
        _ptr(expert_num_tokens, torch.int32, "expert_num_tokens"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream()), "moe_forward_batched_i8")


def selftest_wait_timeout(ws, mode):
    """One bounded wait that nothing satisfies (0: counter, 1: mbarrier); it records ERR_TIMEOUT."""
    _check(lib().moe_selftest_wait_timeout(_ptr(ws, torch.uint8, "ws"), ws.numel(), int(mode), _stream()),
           "moe_selftest_wait_timeout")


def get_error(ws):
    """Synchronises the current stream, returns and clears the device status recorded in ws."""
    v = ctypes.c_int(0)
    _check(lib().moe_get_error(_ptr(ws, torch.uint8, "ws"), _stream(), ctypes.byref(v)), "moe_get_error")
    return int(v.value)
