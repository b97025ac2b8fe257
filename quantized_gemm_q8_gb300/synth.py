"""Seeded synthetic inputs: random GGUF super-blocks, activations and canvases.

This module draws random numbers and lays random bytes into the block
formats; it holds none of the method's arithmetic (no decode, no quantize,
no dot products). Both the CUDA path's tests/bench and the CPU oracle take
their inputs from here.

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used as a counter-based stream:
value i of stream s is mix64(s + (i + 1) * GOLDEN). Normals come from the
Box-Muller transform of two uniforms.

Value ranges (the pages only say "uniform-random"; the plain reading, used by the workloads):
  * every quant bit, every 6-bit Q4_K scale/min and every Q6_K int8 scale is
    uniform over its full range (the raw bytes are uniform);
  * Q4_K d and dmin, and Q6_K d, are f16 values uniform over [2^-14, 2^-13)
    (normal numbers, random 10-bit mantissa, exponent field 1);
  * activations are f32 N(0, 1);
  * the canvas is 20 prompt ids uniform in [0, 126000) followed by the mask id.
A second Q4_K recipe (q4k_blocks_centered) gives zero-centred weights for the commit-parity
tests, where a multi-layer model must keep its masked positions apart.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

QK = 256                 # values per super-block
Q4K_BYTES = 144          # GGUF Q4_K block: f16 d, f16 dmin, 12 B scales, 128 B quants
Q6K_BYTES = 210          # GGUF Q6_K block: 128 B ql, 64 B qh, 16 B int8 scales, f16 d
GGML_Q4_K = 12
GGML_Q6_K = 14

# LLaDA-8B facts used for the synthetic workloads.
LLADA = dict(n_layers=32, d_model=4096, n_heads=32, head_dim=128, d_ff=12288,
             vocab=126464, mask_id=126336, eps=1e-5, rope_theta=500000.0)

CONFIG_SEED_BASE = 20261200


def config_seed(c: int) -> int:
    """Seed of workload c (1..5)."""
    return CONFIG_SEED_BASE + int(c)


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def u64_stream(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n SplitMix64 outputs of stream `seed`, starting at counter `offset`."""
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GOLDEN
    return _mix64(z)


def sub_seed(seed: int, tag: str) -> int:
    """Derive an independent stream seed from (seed, tag) via FNV-1a + mix64."""
    h = 0xCBF29CE484222325
    for ch in tag.encode():
        h ^= ch
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    z = np.array([(seed * 0x9E3779B97F4A7C15 + h) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return int(_mix64(z)[0])


def random_bytes(seed: int, n: int) -> np.ndarray:
    words = u64_stream(seed, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def uniform01(seed: int, n: int) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (u64_stream(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int) -> np.ndarray:
    """Standard normal doubles via Box-Muller on consecutive uniform pairs."""
    m = (n + 1) // 2
    w = u64_stream(seed, 2 * m)
    u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n]


def activations(seed: int, rows: int, k: int) -> np.ndarray:
    """f32 [rows, k] ~ N(0, 1)."""
    return normal(seed, rows * k).astype(np.float32).reshape(rows, k)


def _f16_scale_bits(seed: int, n: int) -> np.ndarray:
    """f16 bit patterns uniform over [2^-14, 2^-13): exponent field 1, random mantissa."""
    mant = (u64_stream(seed, n) >> np.uint64(54)).astype(np.uint16)  # 10 random bits
    return (np.uint16(1 << 10) | mant).astype(np.uint16)


def q4k_blocks(seed: int, n: int, k: int) -> np.ndarray:
    """Random GGUF Q4_K matrix [n rows, k/256 blocks, 144 B] (row-major AoS)."""
    assert k % QK == 0
    nb = n * (k // QK)
    blk = random_bytes(sub_seed(seed, "q4k.bytes"), nb * Q4K_BYTES).reshape(nb, Q4K_BYTES)
    d = _f16_scale_bits(sub_seed(seed, "q4k.d"), nb)
    dmin = _f16_scale_bits(sub_seed(seed, "q4k.dmin"), nb)
    blk[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    blk[:, 2:4] = dmin.view(np.uint8).reshape(nb, 2)
    return blk.reshape(n, k // QK, Q4K_BYTES)


def _f16_bits_in(seed: int, n: int, exp_field: int) -> np.ndarray:
    """f16 bit patterns uniform over [2^(e-15), 2^(e-14)): exponent field e, random mantissa."""
    mant = (u64_stream(seed, n) >> np.uint64(54)).astype(np.uint16)
    return (np.uint16(exp_field << 10) | mant).astype(np.uint16)


def q4k_blocks_centered(seed: int, n: int, k: int) -> np.ndarray:
    """Random GGUF Q4_K matrix whose sub-blocks decode to values centred on zero, like trained
    weights (the plain random bytes of q4k_blocks give every weight a positive mean, which drives
    the residual stream of a multi-layer model towards one direction): quant bits uniform, the
    6-bit scales uniform in [1, 8], each min = round(7.5 * scale) with dmin = d (so a weight is
    about d * scale * (q - 7.5)), and d uniform in [2^-11, 2^-10) (normal f16)."""
    assert k % QK == 0
    nb = n * (k // QK)
    blk = random_bytes(sub_seed(seed, "q4kc.bytes"), nb * Q4K_BYTES).reshape(nb, Q4K_BYTES)
    sc = (u64_stream(sub_seed(seed, "q4kc.scales"), nb * 8) % np.uint64(8)).astype(np.int64).reshape(nb, 8) + 1
    mn = np.floor(7.5 * sc + 0.5).astype(np.int64)
    s = np.zeros((nb, 12), np.int64)
    for j in range(4):  # the GGUF 12-byte packing of eight 6-bit scales and eight 6-bit mins
        s[:, j] = (sc[:, j] & 63) | ((sc[:, j + 4] >> 4) << 6)
        s[:, j + 4] = (mn[:, j] & 63) | ((mn[:, j + 4] >> 4) << 6)
        s[:, j + 8] = (sc[:, j + 4] & 15) | ((mn[:, j + 4] & 15) << 4)
    blk[:, 4:16] = s.astype(np.uint8)
    d = _f16_bits_in(sub_seed(seed, "q4kc.d"), nb, 4)
    blk[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    blk[:, 2:4] = d.view(np.uint8).reshape(nb, 2)
    return blk.reshape(n, k // QK, Q4K_BYTES)


def q6k_blocks(seed: int, n: int, k: int) -> np.ndarray:
    """Random GGUF Q6_K matrix [n rows, k/256 blocks, 210 B] (row-major AoS)."""
    assert k % QK == 0
    nb = n * (k // QK)
    blk = random_bytes(sub_seed(seed, "q6k.bytes"), nb * Q6K_BYTES).reshape(nb, Q6K_BYTES)
    d = _f16_scale_bits(sub_seed(seed, "q6k.d"), nb)
    blk[:, 208:210] = d.view(np.uint8).reshape(nb, 2)
    return blk.reshape(n, k // QK, Q6K_BYTES)


def blocks(type_id: int, seed: int, n: int, k: int) -> np.ndarray:
    if type_id == GGML_Q4_K:
        return q4k_blocks(seed, n, k)
    if type_id == GGML_Q6_K:
        return q6k_blocks(seed, n, k)
    raise ValueError(f"unsupported block type {type_id}")


def canvas(seed: int, prompt_len: int = 20, gen_len: int = 128,
           mask_id: int = LLADA["mask_id"], prompt_max: int = 126000) -> np.ndarray:
    """int32 canvas: prompt ids uniform in [0, prompt_max), then gen_len mask ids."""
    ids = (u64_stream(sub_seed(seed, "canvas"), prompt_len) % np.uint64(prompt_max)).astype(np.int32)
    return np.concatenate([ids, np.full(gen_len, mask_id, dtype=np.int32)])


# --- LLaDA-shaped layer / model weights ------------------------------------------------------
# Matrix types of the synthetic workload: Q, K, O, gate, up in Q4_K; V and down in Q6_K;
# output Q6_K; token_embd Q4_K; norm weights f32 = 1.

LAYER_MATS = (  # name, type, rows, cols
    ("wq", GGML_Q4_K, "d_model", "d_model"),
    ("wk", GGML_Q4_K, "d_model", "d_model"),
    ("wv", GGML_Q6_K, "d_model", "d_model"),
    ("wo", GGML_Q4_K, "d_model", "d_model"),
    ("wgate", GGML_Q4_K, "d_ff", "d_model"),
    ("wup", GGML_Q4_K, "d_ff", "d_model"),
    ("wdown", GGML_Q6_K, "d_model", "d_ff"),
)


def layer_weights(seed: int, layer: int, dims: dict | None = None, centered: bool = False) -> dict:
    """Raw GGUF blocks of one layer's seven projections plus f32 norm weights (= 1). centered:
    the Q4_K matrices come from q4k_blocks_centered (Q6_K values are centred already)."""
    dims = dict(LLADA if dims is None else dims)
    out = {}
    for name, t, r, c in LAYER_MATS:
        sd = sub_seed(seed, f"L{layer}.{name}")
        out[name] = q4k_blocks_centered(sd, dims[r], dims[c]) if centered and t == GGML_Q4_K else \
            blocks(t, sd, dims[r], dims[c])
    out["attn_norm"] = np.ones(dims["d_model"], dtype=np.float32)
    out["ffn_norm"] = np.ones(dims["d_model"], dtype=np.float32)
    return out


def head_weights(seed: int, dims: dict | None = None) -> dict:
    dims = dict(LLADA if dims is None else dims)
    return {
        "w_out": q6k_blocks(sub_seed(seed, "output"), dims["vocab"], dims["d_model"]),
        "out_norm": np.ones(dims["d_model"], dtype=np.float32),
    }


def embed_weights(seed: int, dims: dict | None = None, centered: bool = False) -> np.ndarray:
    dims = dict(LLADA if dims is None else dims)
    gen = q4k_blocks_centered if centered else q4k_blocks
    return gen(sub_seed(seed, "token_embd"), dims["vocab"], dims["d_model"])
