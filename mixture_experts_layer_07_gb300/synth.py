"""Seeded synthetic inputs for the MoE layer.

This module only draws random tensors and rounds them to their storage dtype.
It holds none of the layer's arithmetic (no GEMM, routing, permute or combine),
so both the CUDA library's callers and the CPU oracle's callers can take their
inputs from it without sharing any of the method.

The workloads are shaped like the layers the pages measure on (Qwen3-30B-A3B,
GPT-OSS-20B, a 512-expert layer with a fused shared-expert gate, and a
896/1024-expert routing stress case).  Trained weights are not available, so
every tensor is random:

* hidden states ``x``      bf16, N(0, 1)
* gate weight ``wg``       fp32, N(0, 1/H), shape [G, H] (``nn.Linear`` layout)
* expert ``W1``/``W3``     [E, I, H], N(0, 1/H);  ``W2`` [E, H, I], N(0, 1/I)
* shared expert            same recipe with its own intermediate size
* gate bias (GPT-OSS)      +3.0 on experts 0..3, 0 elsewhere
* selection bias           N(0, 0.1) (variance 0.1) for sigmoid+bias routing
* FP8 weights              e4m3 codes with one fp32 scale per 128x128 block,
                           scale = amax(block)/448, code = RNE(w/scale)
* MXFP4 weights            e2m1 codes, two per byte (element 2i in the low
                           nibble), one UE8M0 scale byte per 32 elements of a
                           row: scale 2^(floor(log2 amax) - 2), code =
                           RNE(w/scale) clamped to +-6 (OCP Microscaling)

Two back ends draw the same distributions:

* ``host_inputs``   numpy Philox keyed by (seed, tensor id, expert); exact and
                    platform independent, for the sizes the oracle can take.
* ``device_inputs`` torch's CUDA Philox, for full-size workloads whose expert
                    weights (up to ~90 GB) must never cross the host link.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# tensor ids used as the second Philox key word
TID_X, TID_WG, TID_W1, TID_W3, TID_W2, TID_SW1, TID_SW3, TID_SW2, TID_SELB = range(1, 10)

FP8_BLOCK = 128
FP8_MAX = 448.0  # largest finite e4m3 magnitude
MX_BLOCK = 32    # elements per MXFP4 scale
# e2m1 magnitudes by code 0..7 and the midpoints between neighbours
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)

MODE_SOFTMAX = 0
MODE_SIGMOID_BIAS = 1


@dataclass(frozen=True)
class LayerSpec:
    """Shape and routing policy of one synthetic MoE layer."""

    name: str
    H: int
    E: int
    K: int
    I: int
    mode: int = MODE_SOFTMAX
    routed_scale: float = 1.0
    wdtype: str = "bf16"          # "bf16", "fp8" (e4m3, 128x128 block scales) or
                                  # "mxfp4" (e2m1, a power-of-two scale per 32)
    act: str = "bf16"             # expert-GEMM activations: "bf16", or "fp8" with
                                  # fp8 weights (W8A8: e4m3 per row and 128 columns)
    has_shared: bool = False
    I_shared: int = 0
    hot_experts: tuple = ()       # experts whose gate logit gets ``hot_bias``
    hot_bias: float = 0.0
    sel_bias_var: float = 0.0     # variance of the selection bias (mode 1)
    T_sweep: tuple = field(default=())

    @property
    def G(self) -> int:
        return self.E + (1 if self.has_shared else 0)

    def with_(self, **kw) -> "LayerSpec":
        d = dict(self.__dict__)
        d.update(kw)
        return LayerSpec(**d)


SPECS = {
    "tiny": LayerSpec("tiny", H=256, E=8, K=2, I=128, T_sweep=(16,)),
    "qwen3_30b_a3b": LayerSpec("qwen3_30b_a3b", H=2048, E=128, K=8, I=768,
                               T_sweep=(1, 2, 8, 32, 256, 2048)),
    "gpt_oss_20b": LayerSpec("gpt_oss_20b", H=2880, E=32, K=4, I=2880, wdtype="fp8",
                             hot_experts=(0, 1, 2, 3), hot_bias=3.0,
                             T_sweep=(32, 512, 4096)),
    "shared_gate": LayerSpec("shared_gate", H=2048, E=512, K=10, I=512, has_shared=True,
                             I_shared=512, T_sweep=(1, 4, 64, 1024)),
    "high_expert": LayerSpec("high_expert", H=7168, E=896, K=16, I=2048,
                             mode=MODE_SIGMOID_BIAS, routed_scale=2.5, sel_bias_var=0.1,
                             T_sweep=(512,)),
}


# ----------------------------------------------------------------------------
# dtype rounding (storage formats only)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the 16-bit codes."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 codes to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, tid: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[int(seed), (int(tid) << 32) | int(sub)]))


def _normal(seed, tid, sub, shape, std) -> np.ndarray:
    z = _rng(seed, tid, sub).standard_normal(size=shape, dtype=np.float32)
    return (z * np.float32(std)).astype(np.float32)


def quantize_fp8_block(w: np.ndarray):
    """Quantise one [rows, cols] float32 matrix to e4m3 codes + fp32 block scales.

    scale = amax(block) / 448 (1 for an all-zero block); code = e4m3(w / scale)
    by torch's float8_e4m3fn cast (round to nearest even) on the host.  Returns
    (codes uint8 [rows, cols], scales float32 [ceil(rows/128), ceil(cols/128)]).
    """
    import torch

    rows, cols = w.shape
    rb, cb = math.ceil(rows / FP8_BLOCK), math.ceil(cols / FP8_BLOCK)
    pad = np.zeros((rb * FP8_BLOCK, cb * FP8_BLOCK), dtype=np.float32)
    pad[:rows, :cols] = w
    blk = pad.reshape(rb, FP8_BLOCK, cb, FP8_BLOCK)
    amax = np.abs(blk).max(axis=(1, 3))
    scales = np.where(amax > 0, (amax / np.float32(FP8_MAX)).astype(np.float32),
                      np.float32(1.0)).astype(np.float32)
    q = (blk / scales[:, None, :, None]).astype(np.float32)
    q = np.clip(q, -FP8_MAX, FP8_MAX).reshape(rb * FP8_BLOCK, cb * FP8_BLOCK)[:rows, :cols]
    codes = torch.from_numpy(np.ascontiguousarray(q)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy(), scales


def _e2m1_codes(mag: np.ndarray) -> np.ndarray:
    """Nearest e2m1 code (0..7) of magnitudes, ties to the even code, clamped
    to 6."""
    mid = np.asarray(E2M1_MID, dtype=np.float32)
    pos = np.searchsorted(mid, mag, side="left")
    tie = (pos < len(mid)) & (mid[np.minimum(pos, len(mid) - 1)] == mag) & (pos % 2 == 1)
    return (pos + tie).astype(np.uint8)


def quantize_mxfp4(w: np.ndarray):
    """Quantise one [rows, cols] float32 matrix (cols % 32 == 0) to MXFP4.

    Per 32 consecutive elements of a row: shared exponent
    e = floor(log2(amax)) - 2 (amax = 0: e = -127), scale byte e + 127 clamped
    to [0, 254]; code = sign | e2m1(|w| / 2^e) (round to nearest even, clamped
    to 6).  Returns (packed uint8 [rows, cols/2], scales uint8 [rows, cols/32])."""
    rows, cols = w.shape
    blk = np.ascontiguousarray(w, dtype=np.float32).reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blk).max(axis=2)
    _, ex = np.frexp(amax)              # amax = m * 2^ex, m in [0.5, 1)
    e = np.where(amax > 0, ex - 1 - 2, -127).astype(np.int32)
    sbyte = np.clip(e + 127, 0, 254).astype(np.uint8)
    e = sbyte.astype(np.int32) - 127
    scaled = np.abs(blk) * np.exp2(-e.astype(np.float32))[:, :, None].astype(np.float32)
    code = _e2m1_codes(scaled.astype(np.float32)) | (np.signbit(blk).astype(np.uint8) << 3)
    code = code.reshape(rows, cols)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, sbyte


def quantize_mxfp4_torch(w):
    """quantize_mxfp4 with torch ops (same rule, same bits), for device draws."""
    import torch

    rows, cols = w.shape
    mid = torch.tensor(E2M1_MID, dtype=torch.float32, device=w.device)
    blk = w.to(torch.float32).reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    amax = blk.abs().amax(dim=2)
    _, ex = torch.frexp(amax)
    e = torch.where(amax > 0, ex - 3, torch.full_like(ex, -127)).clamp(-127, 127)
    mag = (blk.abs() * torch.exp2(-e.to(torch.float32))[:, :, None]).contiguous()
    pos = torch.searchsorted(mid, mag, right=False)
    hit = mid[pos.clamp(max=len(E2M1_MID) - 1)] == mag
    code = pos + (hit & (pos < len(E2M1_MID)) & (pos % 2 == 1)).to(pos.dtype)
    code = (code.to(torch.uint8) | (torch.signbit(blk).to(torch.uint8) << 3)).reshape(rows, cols)
    return code[:, 0::2] | (code[:, 1::2] << 4), (e + 127).to(torch.uint8)


# ----------------------------------------------------------------------------
# host back end (numpy Philox)
# ----------------------------------------------------------------------------

def host_inputs(spec: LayerSpec, T: int, seed: int = 0, experts=None, weights: bool = True) -> dict:
    """Draw every tensor of one layer on the host.

    ``experts`` restricts the expert weights to that list of expert indices (the
    other experts' slots stay zero); by default all E experts are drawn.  Each
    expert matrix has its own Philox key, so a subset equals the same slices of
    the full draw.  ``weights=False`` draws only x, the gate and the biases.

    Returned keys (numpy):
      x_bits [T,H] u16 | wg [G,H] f32 | gate_bias [G] f32 or None |
      sel_bias [E] f32 or None |
      bf16: w1_bits [E,I,H], w3_bits [E,I,H], w2_bits [E,H,I] u16
      fp8 : w1_q/w3_q/w2_q u8 and s1/s3/s2 f32 block scales
      shared: sw1_bits [Is,H], sw3_bits [Is,H], sw2_bits [H,Is] u16
    """
    H, E, I, G = spec.H, spec.E, spec.I, spec.G
    out = {"spec": spec, "T": T, "seed": seed}
    out["x_bits"] = f32_to_bf16_bits(_normal(seed, TID_X, 0, (T, H), 1.0))
    out["wg"] = _normal(seed, TID_WG, 0, (G, H), 1.0 / math.sqrt(H))
    if spec.hot_experts:
        gb = np.zeros(G, dtype=np.float32)
        gb[list(spec.hot_experts)] = np.float32(spec.hot_bias)
        out["gate_bias"] = gb
    else:
        out["gate_bias"] = None
    if spec.sel_bias_var > 0:
        out["sel_bias"] = _normal(seed, TID_SELB, 0, (E,), math.sqrt(spec.sel_bias_var))
    else:
        out["sel_bias"] = None

    ex = list(range(E)) if experts is None else list(experts)
    out["experts"] = ex
    if not weights:
        return out
    std1, std2 = 1.0 / math.sqrt(H), 1.0 / math.sqrt(I)
    if spec.wdtype == "bf16":
        for key, tid, shp, std in (("w1_bits", TID_W1, (I, H), std1),
                                   ("w3_bits", TID_W3, (I, H), std1),
                                   ("w2_bits", TID_W2, (H, I), std2)):
            arr = np.zeros((E,) + shp, dtype=np.uint16)
            for e in ex:
                arr[e] = f32_to_bf16_bits(_normal(seed, tid, e, shp, std))
            out[key] = arr
    elif spec.wdtype == "fp8":
        for qk, sk, tid, shp, std in (("w1_q", "s1", TID_W1, (I, H), std1),
                                      ("w3_q", "s3", TID_W3, (I, H), std1),
                                      ("w2_q", "s2", TID_W2, (H, I), std2)):
            q = np.zeros((E,) + shp, dtype=np.uint8)
            s = np.ones((E, math.ceil(shp[0] / FP8_BLOCK), math.ceil(shp[1] / FP8_BLOCK)),
                        dtype=np.float32)
            for e in ex:
                q[e], s[e] = quantize_fp8_block(_normal(seed, tid, e, shp, std))
            out[qk], out[sk] = q, s
    elif spec.wdtype == "mxfp4":
        for qk, sk, tid, shp, std in (("w1_q4", "s1", TID_W1, (I, H), std1),
                                      ("w3_q4", "s3", TID_W3, (I, H), std1),
                                      ("w2_q4", "s2", TID_W2, (H, I), std2)):
            q = np.zeros((E, shp[0], shp[1] // 2), dtype=np.uint8)
            s = np.full((E, shp[0], shp[1] // MX_BLOCK), 127, dtype=np.uint8)
            for e in ex:
                q[e], s[e] = quantize_mxfp4(_normal(seed, tid, e, shp, std))
            out[qk], out[sk] = q, s
    else:
        raise ValueError(spec.wdtype)

    if spec.has_shared:
        Is = spec.I_shared
        out["sw1_bits"] = f32_to_bf16_bits(_normal(seed, TID_SW1, 0, (Is, H), 1.0 / math.sqrt(H)))
        out["sw3_bits"] = f32_to_bf16_bits(_normal(seed, TID_SW3, 0, (Is, H), 1.0 / math.sqrt(H)))
        out["sw2_bits"] = f32_to_bf16_bits(_normal(seed, TID_SW2, 0, (H, Is), 1.0 / math.sqrt(Is)))
    return out


def random_logits(T: int, G: int, seed: int = 0, hot=(), hot_bias=0.0) -> np.ndarray:
    """fp32 logits ~N(0,1) for routing-only cases (plus an optional hot-expert bias)."""
    lg = _normal(seed, 100, 0, (T, G), 1.0)
    if hot:
        lg[:, list(hot)] += np.float32(hot_bias)
    return lg


def random_ids(T: int, K: int, E: int, seed: int = 0) -> np.ndarray:
    """[T,K] int32 expert ids, K distinct experts per token (permute-only cases)."""
    rng = _rng(seed, 101, 0)
    keys = rng.random((T, E))
    return np.argsort(keys, axis=1)[:, :K].astype(np.int32)


# ----------------------------------------------------------------------------
# device back end (torch CUDA Philox) for full-size workloads
# ----------------------------------------------------------------------------

def device_inputs(spec: LayerSpec, T: int, seed: int = 0, device: str = "cuda") -> dict:
    """Draw every tensor of one layer directly in device memory (torch tensors).

    Same distributions as ``host_inputs`` but torch's CUDA generator, so values
    differ from the host draw.  bf16 tensors are torch.bfloat16; FP8 codes are
    torch.uint8 with fp32 block scales.
    """
    import torch

    H, E, I, G = spec.H, spec.E, spec.I, spec.G
    gen = torch.Generator(device=device)

    def normal(tid, shape, std, sub=0, dtype=torch.bfloat16):
        gen.manual_seed((seed * 1_000_003 + tid) * 65_537 + sub)
        return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
                .mul_(std).to(dtype))

    out = {"spec": spec, "T": T, "seed": seed}
    out["x"] = normal(TID_X, (T, H), 1.0)
    out["wg"] = normal(TID_WG, (G, H), 1.0 / math.sqrt(H), dtype=torch.float32)
    if spec.hot_experts:
        gb = torch.zeros(G, dtype=torch.float32, device=device)
        gb[list(spec.hot_experts)] = spec.hot_bias
        out["gate_bias"] = gb
    else:
        out["gate_bias"] = None
    out["sel_bias"] = (normal(TID_SELB, (E,), math.sqrt(spec.sel_bias_var), dtype=torch.float32)
                       if spec.sel_bias_var > 0 else None)

    std1, std2 = 1.0 / math.sqrt(H), 1.0 / math.sqrt(I)
    if spec.wdtype == "bf16":
        for key, tid, shp, std in (("w1", TID_W1, (I, H), std1), ("w3", TID_W3, (I, H), std1),
                                   ("w2", TID_W2, (H, I), std2)):
            w = torch.empty((E,) + shp, dtype=torch.bfloat16, device=device)
            for e in range(E):
                w[e] = normal(tid, shp, std, sub=e)
            out[key] = w
    elif spec.wdtype == "mxfp4":
        for qk, sk, tid, shp, std in (("w1_q4", "s1", TID_W1, (I, H), std1),
                                      ("w3_q4", "s3", TID_W3, (I, H), std1),
                                      ("w2_q4", "s2", TID_W2, (H, I), std2)):
            q = torch.empty((E, shp[0], shp[1] // 2), dtype=torch.uint8, device=device)
            s = torch.empty((E, shp[0], shp[1] // MX_BLOCK), dtype=torch.uint8, device=device)
            for e in range(E):
                q[e], s[e] = quantize_mxfp4_torch(normal(tid, shp, std, sub=e, dtype=torch.float32))
            out[qk], out[sk] = q, s
    else:
        for qk, sk, tid, shp, std in (("w1_q", "s1", TID_W1, (I, H), std1),
                                      ("w3_q", "s3", TID_W3, (I, H), std1),
                                      ("w2_q", "s2", TID_W2, (H, I), std2)):
            rb, cb = math.ceil(shp[0] / FP8_BLOCK), math.ceil(shp[1] / FP8_BLOCK)
            q = torch.empty((E,) + shp, dtype=torch.uint8, device=device)
            s = torch.empty((E, rb, cb), dtype=torch.float32, device=device)
            for e in range(E):
                w = normal(tid, shp, std, sub=e, dtype=torch.float32)
                pad = torch.zeros(rb * FP8_BLOCK, cb * FP8_BLOCK, device=device)
                pad[:shp[0], :shp[1]] = w
                blk = pad.view(rb, FP8_BLOCK, cb, FP8_BLOCK)
                amax = blk.abs().amax(dim=(1, 3))
                sc = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
                qq = (blk / sc[:, None, :, None]).clamp_(-FP8_MAX, FP8_MAX)
                qq = qq.view(rb * FP8_BLOCK, cb * FP8_BLOCK)[:shp[0], :shp[1]]
                q[e] = qq.to(torch.float8_e4m3fn).view(torch.uint8)
                s[e] = sc
            out[qk], out[sk] = q, s
    if spec.has_shared:
        Is = spec.I_shared
        out["sw1"] = normal(TID_SW1, (Is, H), 1.0 / math.sqrt(H))
        out["sw3"] = normal(TID_SW3, (Is, H), 1.0 / math.sqrt(H))
        out["sw2"] = normal(TID_SW2, (H, Is), 1.0 / math.sqrt(Is))
    return out
