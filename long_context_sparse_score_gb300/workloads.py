"""Seeded synthetic inputs for the sparse-decode path.

This module only draws inputs (random KV caches, queries, 32-bit codes made by
random sign projections, sequence lengths); it holds none of the path's own
arithmetic (no scoring, selection or attention). Both the CUDA path and the CPU
oracle receive exactly the tensors built here.

Workloads (decode shapes of the HashAttention and Nectar pages, synthetic data
in place of their LongBench/RULER prompts and model checkpoints):
  1 tiny single head: B=1, 1/1 heads, d=64, n=1024, fp32 q/K/V ~ N(0,1),
    separate random projections W_q, W_k ~ N(0,1) [32, 64]; m=64, S=4, Lw=16
  2 GQA layer (Llama-3-8B shape): B=1, 32/8 heads, d=128, n=32768, bf16 K/V ~ N(0,1);
    queries 0.8 * (a random cached key of the head's KV head) + 0.6 * N(0,1);
    one projection W[g] ~ N(0,1) [32, 128] per KV head for keys and queries;
    m=1024, S=128, Lw=128
  3 long-context batch: as 2 with B=16, n=131072, m=4096, S=128, Lw=256
  4 shared document: one bf16 document of 61440 tokens (batch stride 0), 32
    queries against it, per-query local KV [32, 8, 512, 128] ~ N(0,1) attended
    densely and merged; m=2048, S=128, Lw=0
  5 ragged batch: B=64, 32/8 heads, seq_len ~ U{4096..65536}, m_b = 64 *
    floor((seq_len + 1024) / 2048), S=64, Lw=128 (and a dense run)
Seeds: sub-stream s of workload c draws from torch.Generator(device) seeded
1000*c + s, s = 0 K, 1 V, 2 W, 3 query key choice, 4 query noise, 5 seq_lens,
6 local KV.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

N_BITS = 32


@dataclass
class Workload:
    name: str
    q: torch.Tensor                 # [B, Hq, d] fp32 or bf16
    q_sig: torch.Tensor             # [B, Hq] int32 (bit pattern of the uint32 code)
    k_sig: torch.Tensor             # [Bk, Hkv, n_cap] int32
    K: torch.Tensor                 # [Bk, Hkv, n_cap, d]
    V: torch.Tensor
    seq_lens: torch.Tensor          # [B] int32
    m: int
    n_sink: int
    n_local: int
    m_per_seq: torch.Tensor | None = None
    K_loc: torch.Tensor | None = None   # [B, Hkv, n_loc, d] (shared-document workload)
    V_loc: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def Hkv(self):
        return self.K.shape[1]

    @property
    def d(self):
        return self.q.shape[2]

    @property
    def n_cap(self):
        return self.K.shape[2]

    @property
    def shared(self):
        return self.K.shape[0] == 1 and self.B > 1


def _gen(cfg: int, sub: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1000 * cfg + sub)
    return g


def mlp_weights(cfg: int, Hkv: int, d: int, hidden: int = 128, device="cpu"):
    """Random weights for the MLP signature map d -> hidden -> hidden -> 32 per KV
    head, float32: W ~ N(0, 1/fan_in), biases ~ N(0, 0.1^2). Returns
    (W1 [Hkv, H, d], b1 [Hkv, H], W2 [Hkv, H, H], b2 [Hkv, H], W3 [Hkv, 32, H], b3 [Hkv, 32])."""
    g = _gen(cfg, 7, device)
    shapes = [((Hkv, hidden, d), d), ((Hkv, hidden), 0), ((Hkv, hidden, hidden), hidden), ((Hkv, hidden), 0),
              ((Hkv, N_BITS, hidden), hidden), ((Hkv, N_BITS), 0)]
    out = []
    for shp, fan_in in shapes:
        t = torch.randn(shp, generator=g, device=device, dtype=torch.float32)
        out.append(t / fan_in ** 0.5 if fan_in else 0.1 * t)
    return tuple(out)


def pack_bits(bits: torch.Tensor) -> torch.Tensor:
    """[..., 32] bool -> int32 word with bit j (LSB = 0) = bits[..., j]."""
    w = torch.arange(N_BITS, device=bits.device, dtype=torch.int64)
    v = (bits.to(torch.int64) << w).sum(-1)
    v = torch.where(v >= 2**31, v - 2**32, v)
    return v.to(torch.int32)


def sign_codes(x: torch.Tensor, W: torch.Tensor) -> torch.Tensor:
    """Bits of sign(W x): bit j = 1 iff <W[j], x> > 0 (0 maps to 0). x [..., d], W [32, d]."""
    proj = x.to(torch.float32) @ W.to(torch.float32).t()
    return pack_bits(proj > 0)


def _kv_codes(K: torch.Tensor, W: torch.Tensor) -> torch.Tensor:
    """Codes of every cached key: K [Bk, Hkv, n, d], W [Hkv, 32, d] -> [Bk, Hkv, n]."""
    Bk, Hkv, n, _ = K.shape
    out = torch.empty((Bk, Hkv, n), dtype=torch.int32, device=K.device)
    for b in range(Bk):
        for g in range(Hkv):
            out[b, g] = sign_codes(K[b, g], W[g])
    return out


def _queries_near_keys(K, W, seq_lens, Hq, cfg, device, q_dtype=torch.bfloat16, shared=False):
    """q[b,h] = 0.8 * K[b, h//G, j] + 0.6 * eps with j ~ U[0, seq_len), eps ~ N(0, 1)."""
    B = seq_lens.shape[0]
    Hkv, d = K.shape[1], K.shape[3]
    G = Hq // Hkv
    gj = _gen(cfg, 3, device)
    ge = _gen(cfg, 4, device)
    u = torch.rand((B, Hq), generator=gj, device=device, dtype=torch.float64)
    lens = seq_lens.to(device=device, dtype=torch.float64).view(B, 1)
    j = torch.clamp((u * lens).floor().to(torch.int64), min=0)
    j = torch.minimum(j, (lens.to(torch.int64) - 1).clamp(min=0))
    eps = torch.randn((B, Hq, d), generator=ge, device=device, dtype=torch.float32)
    bi = torch.zeros((B, Hq), dtype=torch.int64, device=device) if shared else \
        torch.arange(B, device=device).view(B, 1).expand(B, Hq)
    gi = (torch.arange(Hq, device=device) // G).view(1, Hq).expand(B, Hq)
    keys = K[bi, gi, j].to(torch.float32)
    q = (0.8 * keys + 0.6 * eps).to(q_dtype)
    q_sig = torch.empty((B, Hq), dtype=torch.int32, device=device)
    for h in range(Hq):
        q_sig[:, h] = sign_codes(q[:, h].to(torch.float32), W[h // G])
    return q, q_sig


def make_gqa(cfg: int, *, B: int, Hq: int, Hkv: int, d: int, n_cap: int, seq_lens, m: int,
             n_sink: int, n_local: int, device="cpu", kv_dtype=torch.bfloat16,
             shared: bool = False, m_per_seq=None, name: str | None = None) -> Workload:
    """The GQA recipe of workloads 2-5 at any size (tests use reduced sizes)."""
    Bk = 1 if shared else B
    K = torch.randn((Bk, Hkv, n_cap, d), generator=_gen(cfg, 0, device), device=device, dtype=kv_dtype)
    V = torch.randn((Bk, Hkv, n_cap, d), generator=_gen(cfg, 1, device), device=device, dtype=kv_dtype)
    W = torch.randn((Hkv, N_BITS, d), generator=_gen(cfg, 2, device), device=device, dtype=torch.float32)
    if isinstance(seq_lens, int):
        seq_lens = torch.full((B,), seq_lens, dtype=torch.int32)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).to(device)
    k_sig = _kv_codes(K, W)
    q, q_sig = _queries_near_keys(K, W, seq_lens, Hq, cfg, device, shared=shared)
    if m_per_seq is not None:
        m_per_seq = torch.as_tensor(m_per_seq, dtype=torch.int32).to(device)
    return Workload(name or f"gqa{cfg}", q, q_sig, k_sig, K, V, seq_lens, m, n_sink, n_local,
                    m_per_seq=m_per_seq)


def make_tiny(device="cpu", n: int = 1024) -> Workload:
    """Workload 1: one head, d=64, fp32, separate query/key projections."""
    cfg = 1
    d = 64
    K = torch.randn((1, 1, n, d), generator=_gen(cfg, 0, device), device=device)
    V = torch.randn((1, 1, n, d), generator=_gen(cfg, 1, device), device=device)
    gw = _gen(cfg, 2, device)
    W_k = torch.randn((N_BITS, d), generator=gw, device=device)
    W_q = torch.randn((N_BITS, d), generator=gw, device=device)
    q = torch.randn((1, 1, d), generator=_gen(cfg, 4, device), device=device)
    k_sig = sign_codes(K[0, 0], W_k).view(1, 1, n)
    q_sig = sign_codes(q[0, 0], W_q).view(1, 1)
    seq_lens = torch.full((1,), n, dtype=torch.int32, device=device)
    return Workload("tiny", q, q_sig, k_sig, K, V, seq_lens, m=64, n_sink=4, n_local=16)


def ragged_lens(B: int, lo: int, hi: int, device="cpu", cfg: int = 5) -> torch.Tensor:
    """Integer-uniform lengths in [lo, hi] (inclusive) from sub-stream 5."""
    return torch.randint(lo, hi + 1, (B,), generator=_gen(cfg, 5, "cpu"), dtype=torch.int64).to(
        torch.int32).to(device)


def ragged_budget(seq_lens: torch.Tensor) -> torch.Tensor:
    """m_b = seq_len / 32 rounded half up to a multiple of 64: 64 * floor((seq_len + 1024) / 2048)."""
    return (64 * ((seq_lens.to(torch.int64) + 1024) // 2048)).to(torch.int32)


def make_workload(cfg: int, device="cpu", scale: float = 1.0) -> Workload:
    """Workload ``cfg`` (1-5) at full size (scale=1) or with token counts scaled down."""
    if cfg == 1:
        return make_tiny(device, n=max(64, int(1024 * scale)))
    if cfg == 2:
        n = max(256, int(32768 * scale))
        return make_gqa(2, B=1, Hq=32, Hkv=8, d=128, n_cap=n, seq_lens=n, m=1024, n_sink=128,
                        n_local=128, device=device, name="gqa-32k")
    if cfg == 3:
        n = max(256, int(131072 * scale))
        B = 16 if scale >= 1.0 else 2
        return make_gqa(3, B=B, Hq=32, Hkv=8, d=128, n_cap=n, seq_lens=n, m=4096, n_sink=128,
                        n_local=256, device=device, name="batch16-128k")
    if cfg == 4:
        n = max(256, int(61440 * scale))
        B = 32 if scale >= 1.0 else 4
        w = make_gqa(4, B=B, Hq=32, Hkv=8, d=128, n_cap=n, seq_lens=n, m=2048, n_sink=128,
                     n_local=0, device=device, shared=True, name="shared-doc-61440")
        gl = _gen(4, 6, device)
        w.K_loc = torch.randn((B, 8, 512, 128), generator=gl, device=device, dtype=torch.bfloat16)
        w.V_loc = torch.randn((B, 8, 512, 128), generator=gl, device=device, dtype=torch.bfloat16)
        return w
    if cfg == 5:
        B = 64 if scale >= 1.0 else 4
        hi = max(4096, int(65536 * scale))
        lo = min(4096, hi)
        lens = ragged_lens(B, lo, hi, device)
        mb = ragged_budget(lens)
        return make_gqa(5, B=B, Hq=32, Hkv=8, d=128, n_cap=hi, seq_lens=lens,
                        m=int(mb.max().item()), n_sink=64, n_local=128, device=device,
                        m_per_seq=mb, name="ragged64")
    raise ValueError(cfg)
