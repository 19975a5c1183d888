"""Seeded synthetic workloads for draft-tree build and verify.

This module only draws random inputs; it holds none of the method's arithmetic.
Both the CUDA path (tests, bench) and the CPU oracle (tests) take their inputs
from here.  Real drafter/target logits need trained models, so the workloads
stand in for the pages' benchmark prompts with the shapes and value
distributions the pages' settings imply: Qwen3's vocabulary (V = 151936), a
16-token diffusion block, Gaussian logits with an optional "confident" spike.

Recipe (per request r, seeds derived from a base seed s = 1000*cfg + 10*r):
  drafter  x[l, v] = scale * N(0, 1), plus +8 on one uniformly drawn token of
           position l with probability p_spike (independently per position);
           stored as bf16 (round to nearest even) or fp32.
  target   row n (the target's next-token logits after tree node n) is drawn
           the same way with spike probability 0.7; the spike token equals the
           drafter's spike token of position depth(n)+1 with probability 0.8
           (when that position has one), else a uniform token.  Rows of
           depth-L nodes and rows past the tree get a uniform spike token.
  uniforms [2, Mmax] fp32 from torch's generator (Philox on CUDA).
  U, Vt    [V, 64] fp32, 0.1 * N(0, 1), seeds 7 and 8.
"""
import dataclasses
import math

import torch

V_QWEN3 = 151936
SPIKE = 8.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "ddtree" | "dartree" | "talon"
    batch: int
    L: int
    V: int
    dtype: str           # "bf16" | "f32"
    scale: float         # noise standard deviation of the logits
    p_spike: float       # probability of the +8 spike per position (< 0: per-request U(0.2, 0.95))
    temperature: float
    K: int = 0           # DDTree / DARTree candidates per position
    B: int = 0           # node budget (non-root)
    W: int = 0           # DARTree layer width
    beta: float = 0.0    # DARTree depth bonus
    R: int = 0           # DARTree Markov rank
    talon_k: int = 0
    mu: float = 0.0
    N: int = 0           # TALON node budget
    cfg: int = 0         # workload family number (seed base)
    markov_norm: bool = False  # DARTree: full-vocabulary normalised correction
    verify_rule: str = ""      # acceptance rule at T=1 ("" = "ratio"; "iter_residual", "target_match")
    H: int = 0                 # heap mode: TDES hidden units (0: the Markov term when R > 0)
    budget_policy: str = "topb"  # DARTree: "uniform" = DARTree (fixed)
    saba_cv: float = 0.0       # SABA per-node verification cost (0: no SABA)
    saba_cf: float = 0.0       # SABA fixed per-round cost

    @property
    def Kc(self):
        if self.mode == "talon":
            return min(self.N, self.V)
        return self.K

    @property
    def max_nodes(self):
        return (self.N if self.mode == "talon" else self.B) + 1

    @property
    def log_mu(self):
        return float(torch.tensor(math.log(self.mu), dtype=torch.float64).float()) if self.mu > 0 else 0.0

    def with_(self, **kw):
        return dataclasses.replace(self, **kw)


def tiny_greedy():
    """Batch 1, L=4, V=32, K=4, B=8, fp32 logits 2*N(0,1) from seed 0, greedy."""
    return Workload("tiny_greedy_L4_V32_K4_B8", "ddtree", 1, 4, 32, "f32", 2.0, 0.0, 0.0,
                    K=4, B=8, cfg=0)


def single_request(B):
    """Batch 1, L=16, V=151936, bf16, K=B in {64, 128, 256}, DDTree, greedy."""
    return Workload("ddtree_b1_L16_V151936_K%d_B%d" % (B, B), "ddtree", 1, 16, V_QWEN3, "bf16",
                    3.0, 0.7, 0.0, K=B, B=B, cfg=1)


def stochastic_batch(batch):
    """Batch in {1, 4, 16}, L=16, V=151936, bf16, B=K=256, T=1."""
    return Workload("ddtree_t1_b%d_L16_V151936_K256_B256" % batch, "ddtree", batch, 16, V_QWEN3,
                    "bf16", 3.0, 0.7, 1.0, K=256, B=256, cfg=2)


def stochastic_rule(batch, rule):
    """The T=1 workload verified with another acceptance rule."""
    return dataclasses.replace(stochastic_batch(batch), verify_rule=rule,
                               name="ddtree_t1_%s_b%d_L16_V151936_K256_B256" % (rule, batch))


def dartree_supertree(beta):
    """Batch 8, L=16, V=151936, W=32, K=16, R=64, beta in {0, -0.5}, B=512, greedy."""
    return Workload("dartree_b8_L16_V151936_W32_K16_B512_beta%g" % beta, "dartree", 8, 16,
                    V_QWEN3, "bf16", 3.0, 0.7, 0.0, K=16, B=512, W=32, beta=beta, R=64, cfg=3)


def dartree_normalised(beta):
    """The DARTree workload with the full-vocabulary normalised correction."""
    return dataclasses.replace(dartree_supertree(beta), markov_norm=True,
                               name="dartree_norm_b8_L16_V151936_W32_K16_B512_beta%g" % beta)


def dartree_normalised_t1(beta=0.0):
    """The normalised DARTree workload verified at T=1 against its own proposal q~."""
    return dataclasses.replace(dartree_normalised(beta), temperature=1.0,
                               name="dartree_norm_t1_b8_L16_V151936_W32_K16_B512_beta%g" % beta)


def dartree_fixed():
    """DARTree (fixed) at the pages' default: b=8, L=16, K=64, B=64 spread as 4 nodes per depth, R=64."""
    return Workload("dartree_fixed_b8_L16_V151936_K64_B64", "dartree", 8, 16, V_QWEN3, "bf16", 3.0, 0.7, 0.0,
                    K=64, B=64, W=4, R=64, budget_policy="uniform", cfg=3)


def ddtree_saba(batch=16):
    """DDTree with SABA budgets (c_verify 0.5, c_fixed 64: B_t = 128 of at most 256), greedy."""
    return Workload("ddtree_saba_b%d_L16_V151936_K256_Bmax256" % batch, "ddtree", batch, 16, V_QWEN3, "bf16",
                    3.0, 0.7, 0.0, K=256, B=256, saba_cv=0.5, saba_cf=64.0, cfg=2)


def heap_markov(norm=False):
    """The DARTree workload's shapes (b=8, L=16, K=16, B=512, R=64) built by the exact
    best-first heap with the Markov correction (no width limit), optionally normalised."""
    return Workload("heap_markov%s_b8_L16_V151936_K16_B512" % ("_norm" if norm else ""), "heap", 8, 16, V_QWEN3,
                    "bf16", 3.0, 0.7, 0.0, K=16, B=512, R=64, markov_norm=norm, cfg=3)


def heap_tdes(H=256):
    """The same shapes with TDES edge scores (H hidden units, synthetic weights)."""
    return Workload("heap_tdes_H%d_b8_L16_V151936_K16_B512" % H, "heap", 8, 16, V_QWEN3, "bf16", 3.0, 0.7, 0.0,
                    K=16, B=512, H=H, cfg=3)


def tdes_weights(V, L, H, device="cpu"):
    """TDES first-layer rows Ap, Ac [V, H], depth rows Dd [L, H]: 0.3 N(0, 1); output
    weights w [H]: N(0, 1/H); b0 = -0.1, s = 0.8; seeds 11-14."""
    Ap = torch.randn((V, H), generator=_gen(11, device), device=device) * 0.3
    Ac = torch.randn((V, H), generator=_gen(12, device), device=device) * 0.3
    Dd = torch.randn((L, H), generator=_gen(13, device), device=device) * 0.3
    w = torch.randn((H,), generator=_gen(14, device), device=device) * (1.0 / math.sqrt(H))
    return Ap, Ac, Dd, w, -0.1, 0.8


def talon_gated(N):
    """Batch 64, L=16, V=151936, spike prob per request U(0.2, 0.95), k=10, mu=0.03."""
    return Workload("talon_b64_L16_V151936_k10_mu0.03_N%d" % N, "talon", 64, 16, V_QWEN3, "bf16",
                    3.0, -1.0, 0.0, talon_k=10, mu=0.03, N=N, cfg=4)


def all_full_size():
    out = [tiny_greedy()]
    out += [single_request(B) for B in (64, 128, 256)]
    out += [stochastic_batch(b) for b in (1, 4, 16)]
    out += [dartree_supertree(b) for b in (0.0, -0.5)]
    out += [talon_gated(N) for N in (60, 1024)]
    return out


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _seed(wl, req, salt):
    return 1000 * wl.cfg + 10 * req + salt


def _store(x, dtype):
    return x.to(torch.bfloat16) if dtype == "bf16" else x.contiguous()


def request_spike_prob(wl, req, device="cpu"):
    if wl.p_spike >= 0:
        return wl.p_spike
    g = _gen(_seed(wl, req, 5), device)
    return float(0.2 + 0.75 * torch.rand(1, generator=g, device=device).item())


def draft_logits(wl, device="cpu", first_req=0, batch=None):
    """Returns (logits [b, L, V] in wl.dtype, spike_tok [b, L] int64, -1 = no spike)."""
    batch = wl.batch if batch is None else batch
    out = torch.empty((batch, wl.L, wl.V), device=device,
                      dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32)
    spikes = torch.full((batch, wl.L), -1, dtype=torch.int64, device=device)
    for i in range(batch):
        req = first_req + i
        g = _gen(_seed(wl, req, 0), device)
        x = torch.randn((wl.L, wl.V), generator=g, device=device, dtype=torch.float32) * wl.scale
        p = request_spike_prob(wl, req, device)
        if p > 0:
            has = torch.rand(wl.L, generator=g, device=device) < p
            tok = torch.randint(0, wl.V, (wl.L,), generator=g, device=device)
            rows = torch.arange(wl.L, device=device)
            x[rows[has], tok[has]] += SPIKE
            spikes[i] = torch.where(has, tok, torch.full_like(tok, -1))
        out[i] = _store(x, wl.dtype)
    return out, spikes


def target_logits(wl, depth, n_nodes, draft_spikes, device="cpu", first_req=0, rows=None):
    """Target logits [b, Mmax, V] for trees whose node depths are ``depth`` [b, Mmax].

    depth / n_nodes / draft_spikes are tensors or arrays on any device; only the
    first n_nodes[i] rows of request i follow the spike-matching rule."""
    Mmax = wl.max_nodes if rows is None else rows
    depth = torch.as_tensor(depth).to(device=device, dtype=torch.int64)
    n_nodes = torch.as_tensor(n_nodes).to(device="cpu", dtype=torch.int64)
    draft_spikes = torch.as_tensor(draft_spikes).to(device=device, dtype=torch.int64)
    batch = depth.shape[0]
    out = torch.empty((batch, Mmax, wl.V), device=device,
                      dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32)
    for i in range(batch):
        req = first_req + i
        g = _gen(_seed(wl, req, 1), device)
        x = torch.randn((Mmax, wl.V), generator=g, device=device, dtype=torch.float32) * wl.scale
        if wl.p_spike != 0:
            has = torch.rand(Mmax, generator=g, device=device) < 0.7
            match = torch.rand(Mmax, generator=g, device=device) < 0.8
            utok = torch.randint(0, wl.V, (Mmax,), generator=g, device=device)
            d = depth[i, :Mmax].clone()
            valid = torch.arange(Mmax, device=device) < int(n_nodes[i])
            d = torch.where(valid & (d >= 0) & (d < wl.L), d, torch.full_like(d, wl.L))
            ds = torch.cat([draft_spikes[i], torch.full((1,), -1, dtype=torch.int64, device=device)])
            dtok = ds[d]
            tok = torch.where(match & (dtok >= 0), dtok, utok)
            rows_ = torch.arange(Mmax, device=device)
            x[rows_[has], tok[has]] += SPIKE
        out[i] = _store(x, wl.dtype)
    return out


def uniforms(wl, device="cpu", first_req=0, batch=None):
    batch = wl.batch if batch is None else batch
    out = torch.empty((batch, 2, wl.max_nodes), device=device, dtype=torch.float32)
    for i in range(batch):
        g = _gen(_seed(wl, first_req + i, 3), device)
        out[i] = torch.rand((2, wl.max_nodes), generator=g, device=device, dtype=torch.float32)
    return out


def markov_tables(V, R, device="cpu"):
    """U, Vt: [V, R] fp32 entries 0.1 * N(0, 1) from seeds 7 and 8."""
    U = torch.randn((V, R), generator=_gen(7, device), device=device, dtype=torch.float32) * 0.1
    Vt = torch.randn((V, R), generator=_gen(8, device), device=device, dtype=torch.float32) * 0.1
    return U, Vt
