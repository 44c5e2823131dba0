"""Seeded synthetic inputs for the OEA MoE decode layer.

This module only makes input bytes.  It holds none of the layer's arithmetic
(no routing, no expert maths) and is the one piece that both sides share:
the CUDA path (through the library's own device-side generator, which
implements the same element function) and the CPU oracle both consume the
values defined here.

Element generator (counter based, so any slice of a tensor can be produced
on its own):

* SplitMix64 (Steele, Lea & Flood, "Fast Splittable Pseudorandom Number
  Generators", OOPSLA 2014).  Element ``i`` of a stream with seed ``s`` is
  the SplitMix64 output number ``i`` for the initial state ``s``:
  ``mix64(s + (i + 1) * 0x9E3779B97F4A7C15)``.
* An approximately normal value is the centred sum of the four 16-bit
  fields of that 64-bit word (an Irwin-Hall sum of four discrete uniforms),
  scaled to the requested standard deviation.  Only integer arithmetic and
  one correctly rounded fp32 multiply are involved, so the host and the
  GPU produce bit-identical values without any transcendental function.
* bf16 tensors are the fp32 value rounded to nearest-even.

Shapes and layouts (row-major, expert index outermost):
``x [B, d]``, ``W_router [N, d]``, ``W_gate [N, F, d]``, ``W_up [N, F, d]``,
``W_down [N, d, F]``, ``router_bias [N]`` (fp32).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1

# Irwin-Hall(4) over 16-bit fields: mean and standard deviation of the sum.
IH_MEAN = 131070                      # 4 * 65535 / 2
IH_SD = math.sqrt((65536.0 ** 2 - 1.0) / 3.0)   # sqrt(4 * (65536^2 - 1) / 12)

# Tensor ids used to derive per-tensor seeds.
T_X, T_ROUTER, T_GATE, T_UP, T_DOWN, T_BIAS = 0, 1, 2, 3, 4, 5


def mix64(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2^64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Outputs ``start .. start+n-1`` of SplitMix64 with initial state ``seed``."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & MASK64) + i * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def tensor_seed(base_seed: int, layer: int, tensor: int, step: int = 0) -> int:
    """Seed of one tensor of one layer (and, for activations, one step)."""
    return mix64(mix64(base_seed * 0x100000001B3 + layer) + tensor * 0x10001 + step * 0x3F1)


def scale_f32(std: float) -> np.float32:
    """fp32 multiplier that maps the centred Irwin-Hall sum to ``std``."""
    return np.float32(std / IH_SD)


def normal_f32(seed: int, n: int, std: float, start: int = 0) -> np.ndarray:
    """Approximately N(0, std^2) fp32 values, elements ``start .. start+n-1``."""
    r = splitmix64(seed, start, n)
    m = np.uint64(0xFFFF)
    s = ((r & m) + ((r >> np.uint64(16)) & m) + ((r >> np.uint64(32)) & m)
         + (r >> np.uint64(48))).astype(np.int64) - IH_MEAN
    return s.astype(np.float32) * scale_f32(std)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest bf16 (ties to even); returned as fp32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    b = ((b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return b.astype(np.uint32).view(np.float32)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of fp32 values that are exactly bf16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def normal(seed: int, shape, std: float, bf16: bool, start: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    v = normal_f32(seed, n, std, start)
    if bf16:
        v = round_bf16(v)
    return v.reshape(shape)


def permutation(seed: int, n: int) -> np.ndarray:
    """Seeded permutation of 0..n-1 (argsort of SplitMix64 keys)."""
    return np.argsort(splitmix64(seed, 0, n), kind="stable")


def zipf_bias(seed: int, N: int, s: float = 1.1) -> np.ndarray:
    """Per-expert router bias = ln of Zipf(s) popularity over a seeded permutation.

    Expert ``e`` gets popularity rank ``r(e) = perm[e] + 1`` and bias
    ``ln(r^-s / sum_r' r'^-s)``.
    """
    r = permutation(seed, N).astype(np.float64) + 1.0
    pi = r ** (-s)
    pi /= (np.arange(1, N + 1, dtype=np.float64) ** (-s)).sum()
    return np.log(pi).astype(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and input recipe of one synthetic MoE decode workload."""
    name: str
    N: int
    k: int
    d: int
    F: int
    B: int
    bf16: bool = True
    zipf: bool = False
    layers: int = 1
    seed: int = 0
    runs: tuple = ()          # (label, mode, k0, p) routing runs
    int4_cold: bool = False   # cold experts INT4 g128 (hot_n kept bf16)
    hot_n: int = 0
    batch_sweep: tuple = ()

    @property
    def expert_bytes(self) -> int:
        return 3 * self.d * self.F * (2 if self.bf16 else 4)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_fp32_n16_k4_d64_f128_b4", N=16, k=4, d=64, F=128, B=4,
                 bf16=False, seed=0,
                 runs=(("topk", "topk", 4, 1.0), ("oea_k0_2_p0.5", "oea", 2, 0.5))),
        Workload("qwen3_30b_a3b_uniform_b16", N=128, k=8, d=2048, F=768, B=16,
                 seed=30, layers=8,
                 runs=(("topk", "topk", 8, 1.0), ("oea_k0_3", "oea", 3, 1.0),
                       ("oea_k0_5", "oea", 5, 1.0))),
        Workload("qwen3_30b_a3b_zipf_sweep", N=128, k=8, d=2048, F=768, B=16,
                 seed=31, zipf=True, layers=8,
                 runs=(("topk", "topk", 8, 1.0), ("oea_k0_5_p0.7", "oea", 5, 0.7)),
                 batch_sweep=(1, 4, 8, 16, 32, 64, 128, 256)),
        Workload("qwen3_235b_a22b_zipf_b64", N=128, k=8, d=4096, F=1536, B=64,
                 seed=235, zipf=True, layers=8,
                 runs=(("topk", "topk", 8, 1.0), ("oea_k0_5_p0.7", "oea", 5, 0.7)),
                 batch_sweep=(16, 64, 256)),
        Workload("qwen3_30b_a3b_mixed_int4_b32", N=128, k=8, d=2048, F=768, B=32,
                 seed=32, zipf=True, layers=1, int4_cold=True, hot_n=32,
                 runs=(("topk", "topk", 8, 1.0), ("oea_k0_5", "oea", 5, 1.0)),
                 batch_sweep=(8, 16, 32)),
    ]
}


def tensor_std(w: Workload, tensor: int) -> float:
    if tensor == T_X:
        return 1.0
    if tensor in (T_ROUTER, T_GATE, T_UP):
        return 1.0 / math.sqrt(w.d)
    if tensor == T_DOWN:
        return 1.0 / math.sqrt(w.F)
    raise ValueError(tensor)


def tensor_shape(w: Workload, tensor: int, B: int | None = None):
    B = w.B if B is None else B
    return {T_X: (B, w.d), T_ROUTER: (w.N, w.d), T_GATE: (w.N, w.F, w.d),
            T_UP: (w.N, w.F, w.d), T_DOWN: (w.N, w.d, w.F)}[tensor]


def make_tensor(w: Workload, layer: int, tensor: int, B: int | None = None,
                step: int = 0) -> np.ndarray:
    """Full host copy of one input tensor (fp32 holding bf16 values if bf16)."""
    seed = tensor_seed(w.seed, layer, tensor, step if tensor == T_X else 0)
    return normal(seed, tensor_shape(w, tensor, B), tensor_std(w, tensor), w.bf16)


def make_expert(w: Workload, layer: int, e: int):
    """Host copy of one expert's (W_gate[e], W_up[e], W_down[e])."""
    out = []
    for t in (T_GATE, T_UP, T_DOWN):
        seed = tensor_seed(w.seed, layer, t)
        n = w.F * w.d
        shape = (w.F, w.d) if t != T_DOWN else (w.d, w.F)
        out.append(normal(seed, shape, tensor_std(w, t), w.bf16, start=e * n))
    return tuple(out)


def make_bias(w: Workload, layer: int) -> np.ndarray | None:
    if not w.zipf:
        return None
    return zipf_bias(tensor_seed(w.seed, layer, T_BIAS), w.N)


def make_layer(w: Workload, layer: int = 0, B: int | None = None, step: int = 0) -> dict:
    """All inputs of one layer as host arrays."""
    return {
        "x": make_tensor(w, layer, T_X, B, step),
        "w_router": make_tensor(w, layer, T_ROUTER),
        "w_gate": make_tensor(w, layer, T_GATE),
        "w_up": make_tensor(w, layer, T_UP),
        "w_down": make_tensor(w, layer, T_DOWN),
        "bias": make_bias(w, layer),
    }


# ---------------------------------------------------------------------------
# INT4 cold-expert format (input preparation for the mixed-precision layer)
# ---------------------------------------------------------------------------
INT4_GROUP = 128     # scale group along the contraction dimension
INT4_CHUNK = 128     # columns per tile chunk: one scale group
INT4_RB_GATE_UP = 64  # rows per chunk of W_gate / W_up
INT4_RB_DOWN = 128    # rows per chunk of W_down


def quantize_int4(w: np.ndarray):
    """Symmetric group-wise INT4 of a [rows][cols] matrix, groups of 128
    columns: s = bf16(max|w| / 7) (nearest even), q = clamp(rint(w / s), -7, 7)
    with rint rounding half to even, q = 0 where s = 0.  Returns (q int8
    [rows][cols], s fp32 [rows][cols/128] holding bf16 values)."""
    w = np.asarray(w, np.float32)
    R, K = w.shape
    g = w.reshape(R, K // INT4_GROUP, INT4_GROUP).astype(np.float64)
    s = round_bf16((np.abs(g).max(axis=2) / 7.0).astype(np.float32))
    sd = s.astype(np.float64)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sd > 0, np.rint(g / np.where(sd > 0, sd, 1.0)), 0.0)
    q = np.clip(q, -7, 7).astype(np.int8).reshape(R, K)
    return q, s


def pack_int4_tiles(q: np.ndarray, s: np.ndarray, rb: int) -> np.ndarray:
    """Tile-contiguous byte image of one quantised matrix.

    The matrix is cut into chunks of `rb` rows x 128 columns (one scale
    group), stored in the order (row block, column group).  A chunk is
    rb*64 bytes of codes (64 per row) followed by rb bf16 scales (one per
    row: the row's scale of that group).  Codes are stored offset by 8
    (q + 8 in 0..15).  Within a row, column c = 8*h + o (word h, offset o)
    is the nibble at bit 4*(o//2) + 16*(o%2) of 32-bit word h, little
    endian: each 16-bit half of a word holds the codes of two adjacent
    columns four bits apart.
    """
    R, K = q.shape
    assert R % rb == 0 and K % INT4_CHUNK == 0 and INT4_CHUNK == INT4_GROUP
    nrb, nkb = R // rb, K // INT4_CHUNK
    code = (q.astype(np.int16) + 8).astype(np.uint32).reshape(R, K // 8, 8)   # words of 8 columns
    shifts = np.array([0, 16, 4, 20, 8, 24, 12, 28], np.uint32)
    words = (code << shifts[None, None, :]).sum(axis=2, dtype=np.uint64).astype(np.uint32)   # [R][K/8]
    words = words.reshape(nrb, rb, nkb, INT4_CHUNK // 8).transpose(0, 2, 1, 3)             # [nrb][nkb][rb][16]
    code_bytes = np.ascontiguousarray(words).astype("<u4").view(np.uint8).reshape(nrb, nkb, rb * 64)
    sb = to_bf16_bits(np.asarray(s, np.float32)).reshape(nrb, rb, nkb).transpose(0, 2, 1)   # [nrb][nkb][rb]
    scale_bytes = np.ascontiguousarray(sb).astype("<u2").view(np.uint8).reshape(nrb, nkb, rb * 2)
    return np.concatenate([code_bytes, scale_bytes], axis=2).reshape(-1)


def int4_expert_bytes(d: int, F: int) -> int:
    """Bytes of one expert's three packed INT4 matrices: half a byte per
    weight and one bf16 scale per row and 128-column group."""
    return 3 * (d * F // 2 + d * F // INT4_GROUP * 2)


def pack_int4_expert(w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray):
    """(gate, up, down) packed images of one expert, and its (q, s) pairs."""
    out, qs = [], []
    for w, rb in ((w_gate, INT4_RB_GATE_UP), (w_up, INT4_RB_GATE_UP), (w_down, INT4_RB_DOWN)):
        q, s = quantize_int4(w)
        qs.append((q, s))
        out.append(pack_int4_tiles(q, s, rb))
    return out, qs


def trace_seed(w: Workload, layer: int, step: int) -> int:
    """Seed of the hidden states of one step of the hotness trace."""
    return tensor_seed(w.seed + 7919, layer, T_X, step)
