"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds shapes, seeds and random draws only; none of the attention
arithmetic lives here.  Both the CUDA path and the CPU oracle are fed from the
same tensors it returns.

Shapes follow the pages' depth-20 model (10 heads of dimension 128, 2048-token
rows; "nanochat" walkthrough, page 4, pretraining section) and the stress
shapes of the sliding-window workloads.  Values are i.i.d. N(0, 1) drawn in
float32 and rounded to bfloat16, in the order q, k, v, dO from one generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

WINDOW_FULL = -1


@dataclass(frozen=True)
class AttnCall:
    """One forward+backward attention call: [B, T, H, D] tensors and a window."""
    B: int
    T: int
    H: int
    D: int
    window: int
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def shape(self):
        return (self.B, self.T, self.H, self.D)


@dataclass(frozen=True)
class Workload:
    name: str
    calls: tuple = field(default_factory=tuple)


def _seed(config_index: int, call: int) -> int:
    return 100 * config_index + call


# Tiny correctness case: the window counts 32 keys including the query itself.
TINY = Workload("tiny B1 H2 T128 D64 W32", (AttnCall(1, 128, 2, 64, 32, 0),))

# Depth-20-like training layer pair: one sliding-window layer and one full-causal layer.
D20_PAIR = Workload("d20 layer pair B16 T2048 H10 D128 W{1024,2048}",
                    (AttnCall(16, 2048, 10, 128, 1024, _seed(1, 0)),
                     AttnCall(16, 2048, 10, 128, 2048, _seed(1, 1))))

# Depth-30-like layer: four consecutive calls alternating local/global windows.
D30_ALT = Workload("d30 alternating B8 T2048 H15 D128 W{512,2048}x2",
                   tuple(AttnCall(8, 2048, 15, 128, w, _seed(2, c))
                         for c, w in enumerate((512, 2048, 512, 2048))))

# Long-context sliding window: work grows with T*W, not T^2.
LONG_SW = Workload("long context B2 T16384 H16 D128 W1024",
                   (AttnCall(2, 16384, 16, 128, 1024, _seed(3, 0)),))

TRAINING_WORKLOADS = (TINY, D20_PAIR, D30_ALT, LONG_SW)


@dataclass(frozen=True)
class DecodeWorkload:
    """Single-token decode over a padded KV cache [N, Tmax, H, D]."""
    name: str
    N: int
    Tmax: int
    H: int
    D: int
    len_lo: int
    len_hi: int          # inclusive
    windows: tuple
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


DECODE = DecodeWorkload("decode N64 H10 D128 Tmax8192 len U[256,8192] W{1024,full}",
                        64, 8192, 10, 128, 256, 8192, (1024, WINDOW_FULL), _seed(4, 0))


@dataclass(frozen=True)
class PrefillWorkload:
    """Tq new tokens appended to each sequence of a padded KV cache [N, Tmax, H, D].

    A sequence's length counts its new tokens (their keys and values are in the cache)."""
    name: str
    N: int
    Tq: int
    Tmax: int
    H: int
    D: int
    len_lo: int
    len_hi: int          # inclusive
    windows: tuple
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# Prompt prefill after earlier turns (the Engine's prefill over a KV cache): 8 sequences, 2048
# new tokens each, total lengths U[2048, 8192], depth-20 heads.
PREFILL = PrefillWorkload("prefill N8 Tq2048 H10 D128 Tmax8192 len U[2048,8192] W{1024,full}",
                          8, 2048, 8192, 10, 128, 2048, 8192, (1024, WINDOW_FULL), _seed(6, 0))


@dataclass(frozen=True)
class VarlenWorkload:
    """Documents packed into fixed-length rows (document-masked attention over packed rows).

    Document lengths are drawn log-normal (median exp(mu) tokens), clipped to [16, T], and laid
    one after another; a document that does not fit in what is left of a row is cut there and
    continues as a new document at the start of the next row."""
    name: str
    rows: int
    T: int
    H: int
    D: int
    mu: float
    sigma: float
    windows: tuple
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The depth-20 training rows, packed with documents of median ~490 tokens.
VARLEN = VarlenWorkload("packed documents 16 rows x 2048 H10 D128 lengths lognormal(6.2, 0.9) W{1024,full}",
                        16, 2048, 10, 128, 6.2, 0.9, (1024, WINDOW_FULL), _seed(7, 0))


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def make_qkvdo(call: AttnCall, device="cpu"):
    """q, k, v, dO of one call, bf16 contiguous [B, T, H, D] on ``device``."""
    g = generator(call.seed, device)
    return tuple(randn_bf16(call.shape, g, device) for _ in range(4))


def make_qkvdo_shape(B, T, H, D, seed, device="cpu"):
    return make_qkvdo(AttnCall(B, T, H, D, WINDOW_FULL, seed), device)


def decode_lens(wl: DecodeWorkload) -> torch.Tensor:
    """Per-sequence cache lengths, uniform integers in [len_lo, len_hi], int32 on the CPU."""
    g = generator(wl.seed, "cpu")
    return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.N,), generator=g, dtype=torch.int64).to(torch.int32)


def make_decode(wl: DecodeWorkload, device="cpu", poison_tail: bool = False):
    """(q [N,H,D], kcache, vcache [N,Tmax,H,D], lens int32 [N]) with lens on ``device``.

    With ``poison_tail`` every cache slot at or beyond a sequence's length holds
    NaN, so a kernel that reads past the end shows it in its output.
    """
    lens = decode_lens(wl)
    g = generator(wl.seed + 1, device)
    q = randn_bf16((wl.N, wl.H, wl.D), g, device)
    kc = randn_bf16((wl.N, wl.Tmax, wl.H, wl.D), g, device)
    vc = randn_bf16((wl.N, wl.Tmax, wl.H, wl.D), g, device)
    if poison_tail:
        pos = torch.arange(wl.Tmax, device=device).view(1, wl.Tmax)
        dead = (pos >= lens.to(device).view(-1, 1)).view(wl.N, wl.Tmax, 1, 1)
        kc.masked_fill_(dead, float("nan"))
        vc.masked_fill_(dead, float("nan"))
    return q, kc, vc, lens.to(device)


def prefill_lens(wl: PrefillWorkload) -> torch.Tensor:
    """Per-sequence cache lengths (new tokens included), uniform in [len_lo, len_hi], int32 on the CPU."""
    g = generator(wl.seed, "cpu")
    return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.N,), generator=g, dtype=torch.int64).to(torch.int32)


def make_prefill(wl: PrefillWorkload, device="cpu"):
    """(q [N,Tq,H,D], kcache, vcache [N,Tmax,H,D], lens int32 [N]) with lens on ``device``."""
    lens = prefill_lens(wl)
    g = generator(wl.seed + 1, device)
    q = randn_bf16((wl.N, wl.Tq, wl.H, wl.D), g, device)
    kc = randn_bf16((wl.N, wl.Tmax, wl.H, wl.D), g, device)
    vc = randn_bf16((wl.N, wl.Tmax, wl.H, wl.D), g, device)
    return q, kc, vc, lens.to(device)


def prefill_pairs(lens, Tq: int, window: int) -> int:
    """Visible (query, key) pairs of a prefill: new token t of a sequence of length L is position
    L - Tq + t and sees min(W, position + 1) keys."""
    total = 0
    for L in (int(x) for x in lens):
        for t in range(Tq):
            i = L - Tq + t
            total += (i + 1) if window <= 0 else min(window, i + 1)
    return total


def varlen_doc_lengths(wl: VarlenWorkload) -> list:
    """Document lengths of the packed rows, in order (they sum to rows * T)."""
    rng = torch.Generator().manual_seed(wl.seed)
    out = []
    for _ in range(wl.rows):
        left = wl.T
        while left > 0:
            x = torch.randn((), generator=rng).item() * wl.sigma + wl.mu
            L = min(max(int(round(math.exp(x))), 16), wl.T)
            L = min(L, left)
            out.append(L)
            left -= L
    return out


def make_varlen(wl: VarlenWorkload, device="cpu"):
    """(q, k, v, dO [total,H,D] bf16, cu_seqlens int32 [n_docs+1] on ``device``, max_seqlen)."""
    lens = varlen_doc_lengths(wl)
    total = wl.rows * wl.T
    g = generator(wl.seed + 1, device)
    q, k, v, dO = (randn_bf16((total, wl.H, wl.D), g, device) for _ in range(4))
    cu = torch.tensor([0] + list(torch.cumsum(torch.tensor(lens), 0).tolist()), dtype=torch.int32, device=device)
    return q, k, v, dO, cu, max(lens)


def pairs_in_window(T: int, window: int) -> int:
    """Number of (query, key) pairs with j <= i and i - j < W in one row of length T."""
    W = T if (window <= 0 or window >= T) else window
    return T * W - W * (W - 1) // 2


def rope_tables(T: int, D: int, base: float = 10000.0, device="cpu"):
    """Rotary tables (cos, sin), fp32 [T, D/2], as a Llama-like model precomputes them: row t, column i
    hold the cosine and sine of t * base^(-2i/D).  Computed in float64 and rounded once to float32; both
    the CUDA path and the oracle receive these same numbers."""
    t = torch.arange(T, dtype=torch.float64).unsqueeze(1)
    inv_freq = base ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)
    ang = t * inv_freq.unsqueeze(0)
    return ang.cos().to(torch.float32).to(device), ang.sin().to(torch.float32).to(device)
