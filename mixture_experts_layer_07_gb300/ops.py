"""ctypes binding of ``libmoe_gb300.so`` -- argument marshalling only.

Each function has the name of the C entry point it calls (without the
``moe_`` prefix), passes tensor data pointers and the current CUDA stream, and
raises ``MoEError`` when the library returns a status other than MOE_OK.
Every step of the layer runs in the library's CUDA kernels; nothing here
computes.  If the library is not built the import of any function raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MODE_SOFTMAX, MODE_SIGMOID_BIAS = 0, 1
W_BF16, W_FP8, W_MXFP4, W8A8_FP8 = 0, 1, 2, 3
DISPATCH_PER_BLOCK, DISPATCH_GLOBAL_AVG, DISPATCH_SIMT, DISPATCH_ONE_LAUNCH, DISPATCH_GEMV = \
    0, 1, 2, 3, 4
VARIANT_SKIP, VARIANT_SKINNY, VARIANT_TILE, VARIANT_SIMT, VARIANT_WIDE = 0, 1, 2, 3, 4
WIDE_MIN_ROWS = 129
DEV_OK, DEV_BAD_EXPERT_ID, DEV_WAIT_TIMEOUT = 0, 1, 2

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_MISALIGNED", 5: "MOE_ERR_CUDA",
          6: "MOE_ERR_DEVICE_STATUS"}

EXPORTS = ["moe_status_string", "moe_default_m_skinny", "moe_block_variant", "moe_router_gemm",
           "moe_topk_route", "moe_permute_scratch_bytes", "moe_permute",
           "moe_grouped_gemm_scratch_bytes", "moe_grouped_gemm_scratch_bytes_ex",
           "moe_grouped_gemm", "moe_unpermute",
           "moe_workspace_bytes", "moe_layer", "moe_workspace_layout", "moe_permute_static",
           "moe_router_tc_scratch_bytes", "moe_router_gemm_tc", "moe_bounded_wait_check"]

PERMUTE_STATIC_SCRATCH_BYTES = 1 << 20


class MoEError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({_lib().moe_status_string(code).decode()})")


class Config(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int),
                ("K", ctypes.c_int), ("I", ctypes.c_int), ("has_shared", ctypes.c_int),
                ("I_shared", ctypes.c_int), ("mode", ctypes.c_int),
                ("routed_scale", ctypes.c_float), ("wdtype", ctypes.c_int),
                ("m_skinny", ctypes.c_int), ("dispatch", ctypes.c_int)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("wg", "gate_bias", "sel_bias", "w1", "w3", "w2", "s1", "s3", "s2",
                 "sw1", "sw3", "sw2")]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("logits", "ids", "weights", "shared_gate", "offsets", "row_to_flat",
                 "flat_to_row", "xp", "hact", "y", "shared_hact", "shared_y", "block_variant",
                 "permute_scratch", "gemm_scratch", "shared_gemm_scratch", "sync", "splitk",
                 "router_split", "total")]


_L = None
_P, _I, _F, _S, _I64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                        ctypes.c_int64)


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                               "(the MoE path has no fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_status_string.argtypes = [_I]
        lib.moe_default_m_skinny.restype = _I
        lib.moe_default_m_skinny.argtypes = []
        lib.moe_block_variant.restype = _I
        lib.moe_block_variant.argtypes = [_I64, _I64, _I, _I, _I, _I]
        sig = {
            "moe_router_gemm": [_P, _P, _P, _P, _I, _I, _I, _P],
            "moe_router_tc_scratch_bytes": [_I, _I, ctypes.POINTER(_S)],
            "moe_router_gemm_tc": [_P, _P, _P, _P, _I, _I, _I, _P, _S, _P, _P],
            "moe_topk_route": [_P, _I, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P],
            "moe_permute_scratch_bytes": [_I, _I, _I, ctypes.POINTER(_S)],
            "moe_permute": [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P, _P],
            "moe_permute_static": [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P],
            "moe_grouped_gemm_scratch_bytes": [_I, _I, ctypes.POINTER(_S)],
            "moe_grouped_gemm_scratch_bytes_ex": [_I, _I, _I, _I, _I, ctypes.POINTER(_S)],
            "moe_grouped_gemm": [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I,
                                 _I, _P, _P, _S, _P, _P],
            "moe_unpermute": [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P],
            "moe_workspace_bytes": [ctypes.POINTER(Config), ctypes.POINTER(_S)],
            "moe_workspace_layout": [ctypes.POINTER(Config), ctypes.POINTER(WorkspaceLayout)],
            "moe_layer": [ctypes.POINTER(Config), _I, _P, ctypes.POINTER(Weights), _P, _P, _S,
                          _P, _P],
            "moe_bounded_wait_check": [_P, _I, _I, _P, _P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.restype = _I
            fn.argtypes = args
        _L = lib
    return _L


def lib():
    return _lib()


def _p(t):
    """Device pointer of a tensor (or None / a raw int)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, where):
    if code != 0:
        raise MoEError(code, where)


# ---------------------------------------------------------------- host-only
def status_string(code: int) -> str:
    return _lib().moe_status_string(code).decode()


def default_m_skinny() -> int:
    return _lib().moe_default_m_skinny()


def block_variant(m_size: int, R: int, E: int, m_skinny: int = -1,
                  dispatch: int = DISPATCH_PER_BLOCK, wdtype: int = W_BF16) -> int:
    return _lib().moe_block_variant(m_size, R, E, m_skinny, dispatch, wdtype)


def permute_scratch_bytes(T: int, E: int, K: int) -> int:
    n = _S()
    _check(_lib().moe_permute_scratch_bytes(T, E, K, ctypes.byref(n)), "moe_permute_scratch_bytes")
    return n.value


def grouped_gemm_scratch_bytes(R: int, E_blocks: int, H: int = 0, I: int = 0,
                               wdtype: int = W_BF16) -> int:
    n = _S()
    if wdtype == W8A8_FP8:
        _check(_lib().moe_grouped_gemm_scratch_bytes_ex(R, E_blocks, H, I, wdtype,
                                                        ctypes.byref(n)),
               "moe_grouped_gemm_scratch_bytes_ex")
    else:
        _check(_lib().moe_grouped_gemm_scratch_bytes(R, E_blocks, ctypes.byref(n)),
               "moe_grouped_gemm_scratch_bytes")
    return n.value


def make_config(T_max, H, E, K, I, *, has_shared=False, I_shared=0, mode=MODE_SOFTMAX,
                routed_scale=1.0, wdtype=W_BF16, m_skinny=-1, dispatch=DISPATCH_PER_BLOCK) -> Config:
    return Config(T_max, H, E, K, I, int(has_shared), I_shared, mode, routed_scale, wdtype,
                  m_skinny, dispatch)


def workspace_bytes(cfg: Config) -> int:
    n = _S()
    _check(_lib().moe_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_bytes")
    return n.value


def workspace_layout(cfg: Config) -> WorkspaceLayout:
    L = WorkspaceLayout()
    _check(_lib().moe_workspace_layout(ctypes.byref(cfg), ctypes.byref(L)), "moe_workspace_layout")
    return L


# ---------------------------------------------------------------- stages
def router_gemm(x, wg, gate_bias, logits, stream=None):
    T, H = x.shape
    G = wg.shape[0]
    _check(_lib().moe_router_gemm(_p(x), _p(wg), _p(gate_bias), _p(logits), T, H, G,
                                  _stream(stream)), "moe_router_gemm")


def router_tc_scratch_bytes(H: int, G: int) -> int:
    n = _S()
    _check(_lib().moe_router_tc_scratch_bytes(H, G, ctypes.byref(n)), "moe_router_tc_scratch_bytes")
    return n.value


def router_gemm_tc(x, wg, gate_bias, logits, scratch, dev_status=None, stream=None):
    T, H = x.shape
    G = wg.shape[0]
    _check(_lib().moe_router_gemm_tc(_p(x), _p(wg), _p(gate_bias), _p(logits), T, H, G,
                                     _p(scratch), scratch.numel() * scratch.element_size(),
                                     _p(dev_status), _stream(stream)), "moe_router_gemm_tc")


def topk_route(logits, E, K, mode, scale, ids, weights, sel_bias=None, shared_gate=None,
               stream=None):
    T, ld = logits.shape
    _check(_lib().moe_topk_route(_p(logits), ld, _p(sel_bias), T, E, K, mode, float(scale),
                                 _p(ids), _p(weights), _p(shared_gate), _stream(stream)),
           "moe_topk_route")


def permute(x, ids, E, offsets, row_to_flat, flat_to_row, xp, scratch, dev_status=None,
            stream=None, H=None):
    T, K = ids.shape
    H = x.shape[1] if x is not None else H
    _check(_lib().moe_permute(_p(x), _p(ids), T, H, E, K, _p(offsets), _p(row_to_flat),
                              _p(flat_to_row), _p(xp), _p(scratch), scratch.numel(),
                              _p(dev_status), _stream(stream)), "moe_permute")


def permute_static(x, ids, E, offsets, row_to_flat, flat_to_row, xp, dev_status=None,
                   stream=None, H=None):
    """moe_permute_static: moe_permute with the library's built-in scratch, for
    callers that cannot allocate device memory (see the header)."""
    T, K = ids.shape
    H = x.shape[1] if x is not None else H
    _check(_lib().moe_permute_static(_p(x), _p(ids), T, H, E, K, _p(offsets), _p(row_to_flat),
                                     _p(flat_to_row), _p(xp), _p(dev_status), _stream(stream)),
           "moe_permute_static")


def grouped_gemm(xp, offsets, E_blocks, H, I, w1, w3, w2, hact, y, scratch, *, wdtype=W_BF16,
                 s1=None, s3=None, s2=None, m_skinny=-1, dispatch=DISPATCH_PER_BLOCK,
                 block_variant=None, dev_status=None, stream=None, R=None):
    R = xp.shape[0] if R is None else R
    _check(_lib().moe_grouped_gemm(_p(xp), _p(offsets), E_blocks, R, H, I, wdtype, _p(w1),
                                   _p(w3), _p(w2), _p(s1), _p(s3), _p(s2), _p(hact), _p(y),
                                   m_skinny, dispatch, _p(block_variant), _p(scratch),
                                   scratch.numel(), _p(dev_status), _stream(stream)),
           "moe_grouped_gemm")


def unpermute(y, flat_to_row, weights, T, K, H, out, shared_y=None, shared_gate=None,
              stream=None):
    _check(_lib().moe_unpermute(_p(y), _p(flat_to_row), _p(weights), T, K, H, _p(shared_y),
                                _p(shared_gate), _p(out), _stream(stream)), "moe_unpermute")


def layer(cfg: Config, x, weights: Weights, out, workspace, dev_status=None, stream=None, T=None):
    T = x.shape[0] if T is None else T
    _check(_lib().moe_layer(ctypes.byref(cfg), T, _p(x), ctypes.byref(weights), _p(out),
                            _p(workspace), workspace.numel(), _p(dev_status), _stream(stream)),
           "moe_layer")


class MoELayer:
    """Owns the config, the device workspace and the weight pointers of one
    layer and calls ``moe_layer``.  Tensors are kept referenced so their
    pointers stay valid."""

    def __init__(self, cfg: Config, tensors: dict, device="cuda"):
        self.cfg = cfg
        self.tensors = tensors
        g = tensors.get
        self.weights = Weights(*[_p(g(k)) for k in ("wg", "gate_bias", "sel_bias", "w1", "w3",
                                                     "w2", "s1", "s3", "s2", "sw1", "sw3", "sw2")])
        self.workspace = torch.empty(workspace_bytes(cfg), dtype=torch.uint8, device=device)
        self.layout = workspace_layout(cfg)
        # the sync region (up to the logits) starts at zero; see moe_layer
        self.workspace[self.layout.sync:self.layout.logits].zero_()
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)

    def __call__(self, x, out=None, stream=None):
        if out is None:
            out = torch.empty_like(x)
        layer(self.cfg, x, self.weights, out, self.workspace, self.dev_status, stream)
        return out

    def view(self, name, dtype, shape):
        """A typed view of one intermediate inside the workspace."""
        off = getattr(self.layout, name)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype).view(*shape)


def bounded_wait_check(counter, target, limit_us, dev_status, stream=None):
    _check(_lib().moe_bounded_wait_check(_p(counter), target, limit_us, _p(dev_status),
                                         _stream(stream)), "moe_bounded_wait_check")
