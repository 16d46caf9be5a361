"""Seeded synthetic workloads (Llama-3.1-8B attention shapes) shared by the
tests and the benchmark.

This module only draws random inputs; it holds none of the method's
arithmetic.  The pages measure on PG-19 / Ruler with trained Llama-3.1-8B
weights; neither is available, so every tensor here is synthetic with the
shapes of Llama-3.1-8B attention (32 query heads, 8 KV heads, head_dim 128,
vocab 128256) and these value distributions:
  * Q, window queries, K, V ~ N(0, 1);
  * heavy hitters: per (sequence, KV head) exactly round(0.01 * L_b) distinct
    positions in [0, L_b), drawn without replacement, get their K row scaled
    by 8 (exact in bf16); V is unchanged;
  * target logits ~ sigma * N(0, 1) (standard deviation sigma), draft logits
    = target + sigma_n * N(0, 1), or independent sigma * N(0, 1) when
    sigma_n is None;
  * uniforms u ~ U[0, 1), three per position.
Every tensor has its own sub-seed derived from (seed, tensor id, layer).
"""
import torch

# Draft-logit noise of the 32-layer round workload: the value at which the mean
# acceptance sum_x min(p, q) of its seeded logits is 0.9, found by bisection with
# the float64 oracle (tests/golden/calibrate_round_sigma.py -> round_sigma.json).
ROUND_SIGMA_N = 0.25557936727955166

# Workloads by name; each entry's "name" repeats its key.
WORKLOADS = {
    "tiny_b2": dict(name="tiny_b2", B=2, Hq=4, Hkv=1, D=64, dtype="f32", lens=[512, 300], gamma=3, W=16, pool=5, K=64,
            V=1000, sigma=2.0, sigma_n=None, hh=0.0),
    "b32_ctx8k": dict(name="b32_ctx8k", B=32, Hq=32, Hkv=8, D=128, dtype="bf16", lens=8192, gamma=3, W=32, pool=7, K=512,
            V=128256, sigma=3.0, sigma_n=0.5, hh=0.01),
    "b128_ctx32k": dict(name="b128_ctx32k", B=128, Hq=32, Hkv=8, D=128, dtype="bf16", lens=32768, gamma=4, W=32, pool=7,
            K=1024, V=128256, sigma=3.0, sigma_n=0.5, hh=0.01),
    "ragged_b256_ctx4k_64k": dict(name="ragged_b256_ctx4k_64k", B=256, Hq=32, Hkv=8, D=128, dtype="bf16", lens=(4096, 65536), gamma=2,
            W=32, pool=7, K=512, V=128256, sigma=3.0, sigma_n=0.5, hh=0.01),
    "round_b32_ctx16k_32layers": dict(name="round_b32_ctx16k_32layers", B=32, Hq=32, Hkv=8, D=128, dtype="bf16", lens=16384, gamma=3, W=32,
            pool=7, K=512, V=128256, sigma=3.0, sigma_n=ROUND_SIGMA_N, hh=0.01, layers=32),
}

_IDS = dict(k=1, v=2, q=3, qw=4, qd=5, hh=6, tl=7, dl=8, u=9, len=10, mask=11)


def sub_seed(seed, name, layer=0):
    return (seed * 1_000_003 + _IDS[name] * 7_919 + layer * 104_729) % (2 ** 62)


def _gen(device, seed, name, layer=0):
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, name, layer))
    return g


def torch_dtype(cfg):
    return torch.float32 if cfg["dtype"] == "f32" else torch.bfloat16


def lengths(cfg, seed=0):
    """kv_len [B] int32 on the CPU (total cached rows, verify rows included)."""
    B, lens = cfg["B"], cfg["lens"]
    if isinstance(lens, list):
        return torch.tensor(lens, dtype=torch.int32)
    if isinstance(lens, tuple):
        lo, hi = lens
        return torch.randint(lo, hi + 1, (B,), generator=_gen("cpu", seed, "len"), dtype=torch.int64).to(torch.int32)
    return torch.full((B,), lens, dtype=torch.int32)


def capacity(cfg, seed=0):
    lens = cfg["lens"]
    if isinstance(lens, tuple):
        return lens[1]
    return int(lengths(cfg, seed).max())


def kv_cache(cfg, device, seed=0, layer=0, kv_len=None, cap=None):
    """K, V [B, Hkv, cap, D] with heavy-hitter key rows (see module docstring)."""
    B, Hkv, D = cfg["B"], cfg["Hkv"], cfg["D"]
    dt = torch_dtype(cfg)
    if kv_len is None:
        kv_len = lengths(cfg, seed)
    cap = capacity(cfg, seed) if cap is None else cap
    k = torch.randn((B, Hkv, cap, D), generator=_gen(device, seed, "k", layer), device=device, dtype=dt)
    v = torch.randn((B, Hkv, cap, D), generator=_gen(device, seed, "v", layer), device=device, dtype=dt)
    if cfg["hh"] > 0:
        n_hh = torch.round(kv_len.double() * cfg["hh"]).long()          # [B]
        n_max = int(n_hh.max())
        if n_max > 0:
            key = torch.rand((B, Hkv, cap), generator=_gen(device, seed, "hh", layer), device=device)
            pos = torch.arange(cap, device=device)
            key = torch.where(pos[None, None, :] < kv_len.to(device).long()[:, None, None], key,
                              torch.full_like(key, 2.0))
            idx = torch.topk(key, n_max, dim=-1, largest=False, sorted=True).indices   # [B, Hkv, n_max]
            keep = (torch.arange(n_max, device=device)[None, None, :] < n_hh.to(device)[:, None, None]).expand_as(idx)
            bi = torch.arange(B, device=device)[:, None, None].expand_as(idx)[keep]
            hi = torch.arange(Hkv, device=device)[None, :, None].expand_as(idx)[keep]
            ji = idx[keep]
            k[bi, hi, ji] = k[bi, hi, ji] * 8
    return k, v


def queries(cfg, device, seed=0, layer=0, T=None):
    """Verify queries [B, T, Hq, D] with T = gamma + 1 by default."""
    T = cfg["gamma"] + 1 if T is None else T
    return torch.randn((cfg["B"], T, cfg["Hq"], cfg["D"]), generator=_gen(device, seed, "q", layer), device=device,
                       dtype=torch_dtype(cfg))


def window_queries(cfg, device, seed=0, layer=0):
    """SnapKV observation-window queries [B, W, Hq, D]."""
    return torch.randn((cfg["B"], cfg["W"], cfg["Hq"], cfg["D"]), generator=_gen(device, seed, "qw", layer),
                       device=device, dtype=torch_dtype(cfg))


def draft_queries(cfg, device, seed=0, layer=0, step=0):
    """Draft-step queries [B, 1, Hq, D]."""
    return torch.randn((cfg["B"], 1, cfg["Hq"], cfg["D"]), generator=_gen(device, seed, "qd", layer * 64 + step),
                       device=device, dtype=torch_dtype(cfg))


def logits(cfg, device, seed=0, sigma_n="cfg"):
    """(target [B, gamma+1, V], draft [B, gamma, V]) float32.  With cfg["mask_frac"] = m, a seeded
    fraction m of each sequence's vocabulary is -inf in all its rows (a constrained vocabulary),
    and a further 2 % in its target rows only (entries the draft may propose but the target
    forbids)."""
    B, g, V = cfg["B"], cfg["gamma"], cfg["V"]
    sn = cfg["sigma_n"] if sigma_n == "cfg" else sigma_n
    t = torch.randn((B, g + 1, V), generator=_gen(device, seed, "tl"), device=device) * cfg["sigma"]
    noise = torch.randn((B, g, V), generator=_gen(device, seed, "dl"), device=device)
    m = cfg.get("mask_frac")
    if m:
        gm = _gen(device, seed, "mask")
        shared = torch.rand((B, 1, V), generator=gm, device=device) < m
        target_only = torch.rand((B, 1, V), generator=gm, device=device) < 0.02
        t = t.masked_fill(shared, float("-inf"))
    if sn is None:
        d = noise * cfg["sigma"]
        if m:
            d = d.masked_fill(shared, float("-inf"))
    else:
        d = t[:, :g] + noise * sn
    if m:
        t = t.masked_fill(target_only, float("-inf"))
    return t, d.contiguous()


def uniforms(cfg, device, seed=0):
    """u [B, gamma+1, 3] float32 in [0, 1)."""
    u = torch.rand((cfg["B"], cfg["gamma"] + 1, 3), generator=_gen("cpu", seed, "u"))
    return u.to(device)
