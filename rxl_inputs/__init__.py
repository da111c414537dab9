"""Seeded synthetic inputs for relative-position memory attention.

This module is shared by the tests, the benchmark and the oracle harness. It
holds no attention arithmetic: it only draws numbers, rounds them to the
storage type and lays them out. Every element is a pure function of
(seed, tensor id, flat index), so any slice can be regenerated on its own.

Generator
---------
* splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state_n = key + (n+1)*0x9E3779B97F4A7C15,
  output = mix(state_n) with the published finaliser constants.
* uniform in (0, 1): (output >> 11 + 0.5) * 2**-53.
* normals: Box-Muller on consecutive uniform pairs, in float64.
* storage: float64 -> float32 (round to nearest), then, for bf16 workloads,
  float32 -> bf16 with round-to-nearest-even on the bit pattern.

Relative-distance table R
-------------------------
The pages call R a sinusoidal embedding of the distance i-j, projected per
head (Transformer-XL, "Relative Positional Encoding"; the Polish glossary page
names it sinusoidal). The sinusoid itself is not printed on the pages; this
module uses the usual form e_p = [sin(p w_k) | cos(p w_k)], w_k =
10000**(-2k/D), k < D/2, and R_h = E W_R[:, h*dh:(h+1)*dh], computed in
float64 before rounding. R is an input to the attention path, so the choice
does not affect parity.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# tensor ids (fixed; per-segment/per-layer tensors are offset from these)
TID = {"q": 1, "k": 2, "v": 3, "u": 4, "vb": 5, "w_r": 6, "do": 7}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _C1
    z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> np.uint64:
    """Key of one tensor's stream: mix of (seed << 32) + tensor_id."""
    with np.errstate(over="ignore"):
        z = np.array([(int(seed) << 32) + int(tensor_id)], dtype=np.uint64)
        return _mix(z)[0]


def splitmix64(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the tensor's splitmix64 stream."""
    key = stream_key(seed, tensor_id)
    with np.errstate(over="ignore"):
        n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(key + n * GOLDEN)


def uniform(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    z = splitmix64(seed, tensor_id, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, tensor_id: int, shape, std: float = 1.0) -> np.ndarray:
    """float64 N(0, std^2) tensor of `shape` by Box-Muller, chunked."""
    total = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(total, dtype=np.float64)
    pos = 0
    while pos < total:
        n = min(_CHUNK, total - pos)
        npairs = (n + 1) // 2
        p0 = pos // 2  # pos is always even: chunks are even-sized
        u = uniform(seed, tensor_id, 2 * p0, 2 * npairs)
        rad = np.sqrt(-2.0 * np.log(u[0::2]))
        ang = (2.0 * math.pi) * u[1::2]
        pair = np.empty(2 * npairs, dtype=np.float64)
        pair[0::2] = rad * np.cos(ang)
        pair[1::2] = rad * np.sin(ang)
        out[pos:pos + n] = pair[:n]
        pos += n
    return (out * std).reshape(shape)


# ---------------------------------------------------------------- storage types

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round-to-nearest-even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float64 array to the storage dtype; returns float32 values
    (exactly representable in that dtype)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return f
    if dtype == "bf16":
        return bf16_bits_to_f32(f32_to_bf16_bits(f))
    raise ValueError(dtype)


# ----------------------------------------------------------------- R synthesis

def sinusoid(n_pos: int, D: int) -> np.ndarray:
    """[n_pos, D] float64: row p = [sin(p w_k) | cos(p w_k)], w_k = 1e4^(-2k/D)."""
    p = np.arange(n_pos, dtype=np.float64)[:, None]
    k = np.arange(D // 2, dtype=np.float64)[None, :]
    w = 10000.0 ** (-2.0 * k / D)
    return np.concatenate([np.sin(p * w), np.cos(p * w)], axis=1)


def rel_table(n_dist: int, D: int, H: int, dh: int, seed: int, tensor_id: int) -> np.ndarray:
    """[H, n_dist, dh] float64: sinusoid of distances 0..n_dist-1 times a
    random W_R ~ N(0, 1/D) (variance 1/D), split per head."""
    w_r = normal(seed, tensor_id, (D, H * dh), std=1.0 / math.sqrt(D))
    e = sinusoid(n_dist, D) @ w_r
    return np.ascontiguousarray(e.reshape(n_dist, H, dh).transpose(1, 0, 2))


# ------------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    """Shape and distributions of one synthetic workload."""
    name: str
    dtype: str            # "f32" or "bf16"
    B: int
    H: int
    L: int
    M: int                # memory capacity (mem_cap)
    dh: int = 64
    D_model: int = 0      # width of the sinusoid fed to W_R
    segments: int = 1
    layers: int = 1
    backward: bool = True
    mem_start_full: bool = True   # memory already holds M rows on segment 0
    seed: int = 0
    notes: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dh)

    @property
    def n_rel(self) -> int:
        return self.M + self.L


# The five configurations of the path (tiny fp32 case, a 4-segment bf16 stream,
# L=M=512, long memory M=5L, a 16-layer evaluation stream).
CFG1 = Workload("cfg1_f32_B1H1_L4M8", "f32", 1, 1, 4, 8, D_model=64,
                notes="single head, 4x12 score matrix, fwd+bwd+one memory update")
CFG2 = Workload("cfg2_bf16_B8H8_L128M128_4seg", "bf16", 8, 8, 128, 128, D_model=512,
                segments=4, mem_start_full=False,
                notes="one layer over 4 segments, memory starts empty, fwd+bwd per segment")
CFG3 = Workload("cfg3_bf16_B16H16_L512M512", "bf16", 16, 16, 512, 512, D_model=1024,
                notes="fwd+bwd of one layer")
CFG4 = Workload("cfg4_bf16_B8H16_L256M1280", "bf16", 8, 16, 256, 1280, D_model=1024,
                notes="long memory M=5L, fwd+bwd of one layer")
CFG5 = Workload("cfg5_bf16_B4H16_L128M1600_16layer_32seg", "bf16", 4, 16, 128, 1600,
                D_model=1024, segments=32, layers=16, backward=False, mem_start_full=False,
                notes="evaluation stream: attention + memory update, fwd only")
CONFIGS = {1: CFG1, 2: CFG2, 3: CFG3, 4: CFG4, 5: CFG5}


def tensor_id(name: str, segment: int = 0, layer: int = 0) -> int:
    """Fixed id per (tensor, segment, layer); u, v, W_R are per layer only."""
    base = TID[name]
    if name in ("u", "vb", "w_r"):
        return base + 16 * (1 + layer)
    return base + 16 * (1 + layer) + 4096 * (1 + segment)


def layer_params(w: Workload, layer: int = 0) -> dict:
    """Per-layer u, v [H, dh] and R [H, M+L, dh], rounded to the storage type
    (float32 arrays holding storage-type values)."""
    u = normal(w.seed, tensor_id("u", 0, layer), (w.H, w.dh), std=0.02)
    vb = normal(w.seed, tensor_id("vb", 0, layer), (w.H, w.dh), std=0.02)
    r = rel_table(w.n_rel, w.D_model, w.H, w.dh, w.seed, tensor_id("w_r", 0, layer))
    return {"u": round_to(u, w.dtype), "vb": round_to(vb, w.dtype), "r": round_to(r, w.dtype)}


def segment_inputs(w: Workload, segment: int = 0, layer: int = 0, with_grad: bool = None) -> dict:
    """Fresh per-(segment, layer) inputs: q [B,H,L,dh], k_cur / v_cur
    [B,H,L,dh] (the rows this segment appends), and dO [B,H,L,dh] when the
    workload runs a backward. All ~N(0,1)/sqrt(dh) except dO ~ N(0,1)."""
    sd = 1.0 / math.sqrt(w.dh)
    shp = (w.B, w.H, w.L, w.dh)
    out = {
        "q": round_to(normal(w.seed, tensor_id("q", segment, layer), shp, sd), w.dtype),
        "k_cur": round_to(normal(w.seed, tensor_id("k", segment, layer), shp, sd), w.dtype),
        "v_cur": round_to(normal(w.seed, tensor_id("v", segment, layer), shp, sd), w.dtype),
    }
    if with_grad is None:
        with_grad = w.backward
    if with_grad:
        out["do"] = round_to(normal(w.seed, tensor_id("do", segment, layer), shp, 1.0), w.dtype)
    return out


def initial_memory(w: Workload, layer: int = 0) -> dict:
    """Memory held before segment 0, logical order (oldest first):
    k_mem / v_mem [B,H,m0,dh], m0 = M when the workload starts full, else 0.
    A full start is drawn as segment -1 of the same stream."""
    m0 = w.M if w.mem_start_full else 0
    sd = 1.0 / math.sqrt(w.dh)
    shp = (w.B, w.H, m0, w.dh)
    return {
        "k_mem": round_to(normal(w.seed, tensor_id("k", 10**6, layer), shp, sd), w.dtype),
        "v_mem": round_to(normal(w.seed, tensor_id("v", 10**6, layer), shp, sd), w.dtype),
    }


def to_storage_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Raw storage array for a device copy: float32 or uint16 bf16 bits."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    return f32_to_bf16_bits(x)
