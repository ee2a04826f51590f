"""Seeded synthetic workloads for the routed-expert FFN layer of a
DeepSeek-V4-Flash-style MoE ("DeepSeek-V4-Flash 284B - Deep-Dive Mathematical &
Kernel Guide", section 1: 256 routed experts, top-6, w_scale 1.5, hash-routed
layers; colibri "DeepSeek V4 target engine", intro and "Memory policy":
routed experts ship as fp4, the dense set as fp8-e4m3 with UE8M0 block
scales, hidden 4096, ~12.6 MB per expert).

What is drawn here, per configuration:

* expert weights: fp32 N(0, std = 1/sqrt(K)) with K the contraction length
  (H for gate/up, I for down), stored the way the experts ship: MXFP4, i.e.
  32-element e2m1 blocks along K, two codes per byte (even element in the low
  nibble) and one UE8M0 scale byte per block, scale 2^(floor(log2 amax) - 2),
  round-to-nearest-even, saturating at +-6;
* or (the NVFP4-style variant, configurations with wfmt "nvfp4"; CISM
  VALIDATION, "4-bit quantization scheme study", row "E2M1 + E4M3 b16") the
  same fp32 draws as e2m1 codes in 16-element blocks along K with one e4m3
  scale per block and one fp32 scale per matrix: g = amax(matrix) / (6 * 448),
  block scale = e4m3(amax(block) / (6 g)) rounded to nearest even, codes
  e2m1(w / (scale * g)) rounded to nearest even, saturating at +-6;
* the optional shared expert: fp32 draws of the same shape stored as fp8 e4m3
  with one UE8M0 scale per 128x128 tile, scale 2^(floor(log2 amax) - 8),
  round-to-nearest-even, saturating at +-448;
* activations: fp32 N(0,1) rounded to bf16 (round-to-nearest-even);
* router logits: fp32 N(0,1) (+ a per-expert bias where the configuration has
  one), with every token row redrawn until its k+1 largest logits are pairwise
  at least LOGIT_GAP apart, so that the top-k set and its order are unique;
* token ids and the token-id -> expert hash table of the hash-routed layers.

Encoding the weights is part of making the inputs: the layer itself only ever
reads MXFP4 / fp8 weights.  Nothing here routes, permutes, quantises
activations or multiplies.

Random streams: numpy PCG64 seeded through SeedSequence(seed) with the
children [weights, shared weights, bias/permutation, logits, x, token ids], in
that order; every expert matrix has its own grandchild stream, so the bytes do
not depend on how many threads generate them.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path
from typing import Optional

import numpy as np

HASH_VOCAB = 129280          # token-id range of the hash-routed layers
LOGIT_GAP = 1e-3             # min gap between adjacent top-(k+1) logits of a row

_STREAMS = ("weights", "shared", "bias", "logits", "x", "tokens")


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    index: int
    name: str
    H: int                   # hidden size
    I: int                   # expert intermediate size
    E: int                   # routed experts
    k: int                   # experts per token
    T: int                   # tokens per layer call
    steps: int = 1           # independent layer calls (decode: one token each)
    router: str = "learned"  # "learned" or "hash"
    bias: Optional[str] = None   # None, "normal0.5", "zipf1.1"
    shared: bool = False
    w_scale: float = 1.5
    wfmt: str = "mxfp4"      # routed-expert weight format: "mxfp4" or "nvfp4"

    @property
    def default_seed(self) -> int:
        """Seed of the per-call inputs (logits, x, token ids)."""
        return 1000 + self.index

    @property
    def weight_seed(self) -> int:
        """Seed of the expert weights: every configuration with the guide's
        full layer shape uses one weight set (that of the decode layer)."""
        return 1000 if (self.H, self.I, self.E) == (256, 128, 16) else 1001


CONFIGS = {
    0: LayerConfig(0, "tiny", H=256, I=128, E=16, k=2, T=4),
    1: LayerConfig(1, "decode_t1", H=4096, I=2048, E=256, k=6, T=1, steps=4096),
    2: LayerConfig(2, "batched_decode_t32_hash", H=4096, I=2048, E=256, k=6, T=32,
                   router="hash"),
    3: LayerConfig(3, "prefill_pp512", H=4096, I=2048, E=256, k=6, T=512,
                   bias="normal0.5"),
    4: LayerConfig(4, "prefill_t8192_zipf_shared", H=4096, I=2048, E=256, k=6, T=8192,
                   bias="zipf1.1", shared=True),
    # the NVFP4-style weight variant of the tiny, decode and pp512 layers
    # (the same fp32 weight draws, encoded as e2m1 + e4m3 per 16 + fp32 per matrix)
    5: LayerConfig(5, "tiny_nvfp4", H=256, I=128, E=16, k=2, T=4, wfmt="nvfp4"),
    6: LayerConfig(6, "decode_t1_nvfp4", H=4096, I=2048, E=256, k=6, T=1, steps=4096, wfmt="nvfp4"),
    7: LayerConfig(7, "prefill_pp512_nvfp4", H=4096, I=2048, E=256, k=6, T=512, bias="normal0.5",
                   wfmt="nvfp4"),
}


# --------------------------------------------------------------------------
# storage formats (encoders used only to build inputs)
# --------------------------------------------------------------------------
# e2m1 magnitudes in code order 0..7 and the midpoints between neighbours.
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
_E2M1_MID = (_E2M1_MAG[1:] + _E2M1_MAG[:-1]) / 2


def _e4m3_magnitudes() -> np.ndarray:
    """Values of the e4m3 (fn) codes 0..126 (0x7f is NaN), increasing."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e - 7.0))
    return v.astype(np.float32)


_E4M3_MAG = _e4m3_magnitudes()
_E4M3_MID = (_E4M3_MAG[1:] + _E4M3_MAG[:-1]) / 2


def _rne_index(mag: np.ndarray, mids: np.ndarray) -> np.ndarray:
    """Index of the nearest grid point, ties to the even index; saturates."""
    idx = np.searchsorted(mids, mag, side="left")
    at = np.minimum(idx, len(mids) - 1)
    tie = (idx < len(mids)) & (mag == mids[at])
    return np.where(tie & (idx % 2 == 1), idx + 1, idx).astype(np.uint8)


def _floor_log2(amax: np.ndarray) -> np.ndarray:
    _, e = np.frexp(amax)
    return e.astype(np.int32) - 1


def _e2m1_index(mag: np.ndarray) -> np.ndarray:
    """Nearest e2m1 magnitude index (0..7), ties to the even index, saturating.

    The grid has step 0.5 on [0, 2], 1 on [2, 4] and 2 on [4, 6]; rint rounds
    ties to even, and an even index is an even mantissa bit.
    """
    lo = np.rint(mag * 2)                     # [0, 2): index 0..4
    mid = np.rint(mag) + 2                    # [2, 4): index 4..6
    hi = np.minimum(np.rint(mag * 0.5) + 4, 7)   # [4, inf): index 6..7
    idx = np.where(mag < 2, lo, np.where(mag < 4, mid, hi))
    return idx.astype(np.uint8)


def encode_mxfp4_rows(w: np.ndarray):
    """fp32 [rows][K] -> (packed e2m1 [rows][K/2] u8, UE8M0 [rows][K/32] u8)."""
    rows, K = w.shape
    b = w.reshape(rows, K // 32, 32)
    amax = np.abs(b).max(axis=2)
    ex = np.where(amax > 0, _floor_log2(amax) - 2, -127)
    ex = np.clip(ex, -127, 127)
    inv = np.ldexp(np.float32(1.0), (-ex).astype(np.int32)).astype(np.float32)
    y = b * inv[..., None]                    # exact: power-of-two scaling
    code = _e2m1_index(np.abs(y)) | (np.signbit(y).astype(np.uint8) << 3)
    code = code.reshape(rows, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, (ex + 127).astype(np.uint8)


def encode_nvfp4_rows(w: np.ndarray):
    """fp32 [rows][K] -> (packed e2m1 [rows][K/2] u8, e4m3 block scales
    [rows][K/16] u8, fp32 matrix scale g).  Element value = e2m1(code) *
    e4m3(scale) * g."""
    rows, K = w.shape
    amax_t = np.float32(np.abs(w).max())
    g = np.float32(amax_t / np.float32(6.0 * 448.0)) if amax_t > 0 else np.float32(1.0)
    b = w.reshape(rows, K // 16, 16)
    target = (np.abs(b).max(axis=2) / np.float32(6.0) / g).astype(np.float32)
    sbyte = _rne_index(target, _E4M3_MID)                  # 0..126, saturating at 448
    denom = (_E4M3_MAG[sbyte] * g).astype(np.float32)
    safe = np.where(denom > 0, denom, np.float32(1.0))
    y = np.where(denom[..., None] > 0, b / safe[..., None], np.float32(0.0)).astype(np.float32)
    code = _e2m1_index(np.abs(y)) | (np.signbit(y).astype(np.uint8) << 3)
    code = code.reshape(rows, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, sbyte.astype(np.uint8), g


def encode_fp8_tiles(w: np.ndarray, tile: int = 128):
    """fp32 [R][C] -> (e4m3 [R][C] u8, UE8M0 [R/tile][C/tile] u8)."""
    R, C = w.shape
    b = w.reshape(R // tile, tile, C // tile, tile)
    amax = np.abs(b).max(axis=(1, 3))
    ex = np.where(amax > 0, _floor_log2(amax) - 8, -127)
    ex = np.clip(ex, -127, 127)
    y = np.ldexp(b, (-ex)[:, None, :, None].astype(np.int32)).astype(np.float32)
    code = _rne_index(np.abs(y), _E4M3_MID) | (np.signbit(y).astype(np.uint8) << 7)
    return code.reshape(R, C).astype(np.uint8), (ex + 127).astype(np.uint8)


def bf16_bits_from_f32(f: np.ndarray) -> np.ndarray:
    """Round finite fp32 to bf16 (nearest, ties to even); returns u16 bits."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    return ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Weights:
    cfg: LayerConfig
    gate_q: np.ndarray   # u8 [E][I][H/2]
    gate_s: np.ndarray   # u8 [E][I][H/32]
    up_q: np.ndarray     # u8 [E][I][H/2]
    up_s: np.ndarray     # u8 [E][I][H/32]
    down_q: np.ndarray   # u8 [E][H][I/2]
    down_s: np.ndarray   # u8 [E][H][I/32]
    sh_gate_q: Optional[np.ndarray] = None   # u8 e4m3 [I][H]
    sh_gate_s: Optional[np.ndarray] = None   # u8 [I/128][H/128]
    sh_up_q: Optional[np.ndarray] = None
    sh_up_s: Optional[np.ndarray] = None
    sh_down_q: Optional[np.ndarray] = None   # u8 e4m3 [H][I]
    sh_down_s: Optional[np.ndarray] = None   # u8 [H/128][I/128]
    # NVFP4 only: the scales above are e4m3 [E][rows][K/16], plus one fp32
    # scale per expert matrix
    gate_g: Optional[np.ndarray] = None      # f32 [E]
    up_g: Optional[np.ndarray] = None
    down_g: Optional[np.ndarray] = None

    ARRAYS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
              "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q", "sh_down_s",
              "gate_g", "up_g", "down_g")


def _streams(seed: int):
    return dict(zip(_STREAMS, np.random.SeedSequence(seed).spawn(len(_STREAMS))))


def _draw(ss: np.random.SeedSequence, rows: int, K: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(ss))
    w = rng.standard_normal((rows, K), dtype=np.float32)
    w *= np.float32(1.0 / np.sqrt(K))
    return w


def _cache_dir(cfg: LayerConfig, seed: int) -> Optional[Path]:
    root = os.environ.get("BQE_WORKLOAD_CACHE", str(Path.home() / ".cache" / "bqe_workloads"))
    if root in ("", "0", "off"):
        return None
    fmt = "" if cfg.wfmt == "mxfp4" else f"_{cfg.wfmt}"
    return Path(root) / f"H{cfg.H}_I{cfg.I}_E{cfg.E}_s{seed}{fmt}"


def make_weights(cfg: LayerConfig, seed: Optional[int] = None, threads: Optional[int] = None,
                 cache: bool = True) -> Weights:
    """Draw and encode every expert matrix of `cfg` (deterministic in seed)."""
    seed = cfg.weight_seed if seed is None else seed
    if cfg.shared:  # routed experts as without the shared expert, plus its three matrices
        w = make_weights(dataclasses.replace(cfg, shared=False), seed, threads, cache)
        w = dataclasses.replace(w, cfg=cfg)
        sk = _streams(seed)["shared"].spawn(3)
        w.sh_gate_q, w.sh_gate_s = encode_fp8_tiles(_draw(sk[0], cfg.I, cfg.H))
        w.sh_up_q, w.sh_up_s = encode_fp8_tiles(_draw(sk[1], cfg.I, cfg.H))
        w.sh_down_q, w.sh_down_s = encode_fp8_tiles(_draw(sk[2], cfg.H, cfg.I))
        return w
    H, I, E = cfg.H, cfg.I, cfg.E
    big = E * H * I >= (1 << 28)
    cdir = _cache_dir(cfg, seed) if (cache and big) else None
    if cdir is not None and (cdir / "done").exists():
        arrs = {}
        for n in Weights.ARRAYS:
            p = cdir / f"{n}.npy"
            arrs[n] = np.load(p, mmap_mode="r") if p.exists() else None
        return Weights(cfg, **arrs)

    st = _streams(seed)
    kids = st["weights"].spawn(3 * E)
    nv = cfg.wfmt == "nvfp4"
    blk = 16 if nv else 32
    w = Weights(cfg,
                gate_q=np.empty((E, I, H // 2), np.uint8), gate_s=np.empty((E, I, H // blk), np.uint8),
                up_q=np.empty((E, I, H // 2), np.uint8), up_s=np.empty((E, I, H // blk), np.uint8),
                down_q=np.empty((E, H, I // 2), np.uint8), down_s=np.empty((E, H, I // blk), np.uint8))
    if nv:
        w.gate_g, w.up_g, w.down_g = (np.empty(E, np.float32) for _ in range(3))

    def job(i):
        e, m = divmod(i, 3)
        wf = _draw(kids[i], I, H) if m < 2 else _draw(kids[i], H, I)
        if nv:
            q, s, g = encode_nvfp4_rows(wf)
            (w.gate_g, w.up_g, w.down_g)[m][e] = g
        else:
            q, s = encode_mxfp4_rows(wf)
        (w.gate_q, w.up_q, w.down_q)[m][e] = q
        (w.gate_s, w.up_s, w.down_s)[m][e] = s

    nthr = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(nthr) as ex:
        list(ex.map(job, range(3 * E)))

    if cdir is not None:
        try:
            cdir.mkdir(parents=True, exist_ok=True)
            for n in Weights.ARRAYS:
                a = getattr(w, n)
                if a is not None:
                    np.save(cdir / f"{n}.npy", a)
            (cdir / "done").write_text("ok\n")
        except OSError:
            pass
    return w


# --------------------------------------------------------------------------
# per-call inputs
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Tokens:
    x_bits: np.ndarray                  # u16 bf16 bits [n][H]
    logits: np.ndarray                  # f32 [n][E] (bias already added)
    token_ids: Optional[np.ndarray]     # i32 [n] (hash-routed configs)


def _bias(cfg: LayerConfig, st) -> Optional[np.ndarray]:
    rng = np.random.Generator(np.random.PCG64(st["bias"]))
    if cfg.bias is None:
        return None
    if cfg.bias == "normal0.5":
        return (rng.standard_normal(cfg.E) * 0.5).astype(np.float32)
    if cfg.bias == "zipf1.1":
        perm = rng.permutation(cfg.E)
        b = np.empty(cfg.E, np.float64)
        b[perm] = -1.1 * np.log(np.arange(cfg.E) + 1.0)
        return b.astype(np.float32)
    raise ValueError(cfg.bias)


def _row_ok(row: np.ndarray, k: int) -> bool:
    top = np.sort(row)[::-1][: k + 1]
    return bool(np.all(top[:-1] - top[1:] >= LOGIT_GAP))


def make_tokens(cfg: LayerConfig, seed: Optional[int] = None, n: Optional[int] = None) -> Tokens:
    """Inputs for n token rows (default T * steps); row i of a decode run is call i."""
    seed = cfg.default_seed if seed is None else seed
    n = cfg.T * cfg.steps if n is None else n
    st = _streams(seed)
    bias = _bias(cfg, st)
    lrng = np.random.Generator(np.random.PCG64(st["logits"]))
    logits = lrng.standard_normal((n, cfg.E), dtype=np.float32)
    if bias is not None:
        logits += bias[None, :]
    for i in range(n):
        while not _row_ok(logits[i], cfg.k):
            logits[i] = lrng.standard_normal(cfg.E, dtype=np.float32)
            if bias is not None:
                logits[i] += bias
    xrng = np.random.Generator(np.random.PCG64(st["x"]))
    x_bits = bf16_bits_from_f32(xrng.standard_normal((n, cfg.H), dtype=np.float32))
    token_ids = None
    if cfg.router == "hash":
        trng = np.random.Generator(np.random.PCG64(st["tokens"]))
        token_ids = trng.integers(0, HASH_VOCAB, size=n, dtype=np.int64).astype(np.int32)
    return Tokens(x_bits=x_bits, logits=logits, token_ids=token_ids)


def make_hash_table(cfg: LayerConfig, seed: Optional[int] = None,
                    vocab: int = HASH_VOCAB) -> np.ndarray:
    """tid2eid [vocab][k]: k distinct experts per token id (partial Fisher-Yates)."""
    seed = cfg.default_seed if seed is None else seed
    st = _streams(seed)
    rng = np.random.Generator(np.random.PCG64(st["tokens"].spawn(1)[0]))
    perm = np.tile(np.arange(cfg.E, dtype=np.int32), (vocab, 1))
    rows = np.arange(vocab)
    for j in range(cfg.k):
        r = rng.integers(j, cfg.E, size=vocab)
        a, b = perm[rows, j].copy(), perm[rows, r].copy()
        perm[rows, j], perm[rows, r] = b, a
    return np.ascontiguousarray(perm[:, : cfg.k])
