"""Seeded synthetic inputs for the routed-expert MoE layer.

Serves both the CPU oracle and the CUDA library and holds none of the method's arithmetic:
it draws random codes and numbers, prepares activations with torch's own float8/bf16
casts, and picks top-k experts. Weights may be drawn on a CUDA device (torch's generator)
and copied back for the oracle, since a full layer holds 6 GB of expert weights.

Workloads (sizes and distributions of the DeepSeek-class decode and prompt-chunk layers):
  tiny    H 256,  I 128,  E 8,   k 2, R 4,    bf16 activations, random top-2 routing
  decode  H 7168, I 2048, E 256, k 8, R 1,    E4M3 activations (per-32 E8M0 scales)
  shared  decode widths, R in {2,3,4,5,8,16}, every row on the same 8 experts, E4M3
  apart   decode widths, R in {2,4,8,16},     independent random top-8 per row, bf16
  chunk   decode widths, R 4096,              independent random top-8 per row, E4M3
Weights: E2M1 codes uniform over all 16 codes (uniform bytes), one E8M0 scale per 32
k-elements with exponent uniform in [-4, 2] (codes 123..129). Activations: N(0, 1) before
conversion. Routing weights: softmax over the k selected logits.
"""
import numpy as np

ACT_E4M3 = 0
ACT_BF16 = 1

SEED_BASE = 0x7F4E0000

WORKLOADS = {
    "tiny": dict(H=256, I=128, E=8, k=2, R=4, kind=ACT_BF16, routing="random", index=0),
    "decode": dict(H=7168, I=2048, E=256, k=8, R=1, kind=ACT_E4M3, routing="random", index=1),
    "shared": dict(H=7168, I=2048, E=256, k=8, R=4, kind=ACT_E4M3, routing="shared", index=2),
    "apart": dict(H=7168, I=2048, E=256, k=8, R=4, kind=ACT_BF16, routing="random", index=3),
    "chunk": dict(H=7168, I=2048, E=256, k=8, R=4096, kind=ACT_E4M3, routing="random", index=4),
}


def workload(name, **over):
    cfg = dict(WORKLOADS[name])
    cfg.update(over)
    cfg["name"] = name
    cfg.setdefault("seed", SEED_BASE + cfg["index"])
    return cfg


# ------------------------------------------------------------------ weights

def weight_shapes(E, H, I):
    return dict(wg=(E, I, H // 2), sg=(E, I, H // 32), wu=(E, I, H // 2), su=(E, I, H // 32),
                wd=(E, H, I // 2), sd=(E, H, I // 32))


def weights_numpy(E, H, I, seed, scale_lo=123, scale_hi=129):
    """Canonical-layout expert weights as numpy uint8 arrays."""
    rng = np.random.default_rng(seed)
    out = {}
    for name, shp in weight_shapes(E, H, I).items():
        if name.startswith("w"):
            out[name] = rng.integers(0, 256, size=shp, dtype=np.uint8)
        else:
            out[name] = rng.integers(scale_lo, scale_hi + 1, size=shp, dtype=np.uint8)
    return out


def weights_torch(E, H, I, seed, device, scale_lo=123, scale_hi=129):
    """The same distributions drawn on a torch device (a CUDA device for full-size layers)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = {}
    for name, shp in weight_shapes(E, H, I).items():
        if name.startswith("w"):
            out[name] = torch.randint(0, 256, shp, generator=gen, dtype=torch.uint8, device=device)
        else:
            out[name] = torch.randint(scale_lo, scale_hi + 1, shp, generator=gen, dtype=torch.uint8, device=device)
    return out


# ------------------------------------------------------------------ activations

def activations(z, kind):
    """Convert fp32 activations [R, K] to the launch format.

    E4M3: per 32 consecutive values one E8M0 scale 2^(floor(log2 amax) - 8) (the OCP MX
    choice), values divided by it, clamped to +-448 and cast by torch to float8_e4m3fn.
    bf16: torch's cast. Returns (x, sx) with sx None for bf16.
    """
    import torch
    z = np.ascontiguousarray(z, np.float32)
    R, K = z.shape
    if kind == ACT_BF16:
        x = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return np.ascontiguousarray(x), None
    blocks = z.reshape(R, K // 32, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    _, e2 = np.frexp(amax)
    sc = np.where(amax > 0, np.clip(e2 - 1 - 8 + 127, 0, 254), 127).astype(np.int64)
    v = blocks / np.exp2(sc - 127)[:, :, None]
    v = np.clip(v, -448.0, 448.0).reshape(R, K).astype(np.float32)
    x = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.ascontiguousarray(x), sc.astype(np.uint8)


# ------------------------------------------------------------------ routing

def _softmax(l):
    l = l.astype(np.float64)
    m = l.max(axis=1, keepdims=True)
    p = np.exp(l - m)
    return (p / p.sum(axis=1, keepdims=True)).astype(np.float32)


def routing(rng, R, E, k, mode):
    """ids [R, k] int32 (slot order = descending logit, ties to the lower id) and softmax weights."""
    if mode == "shared":
        experts = np.sort(rng.choice(E, size=k, replace=False))
        logits = rng.standard_normal((R, k)).astype(np.float32)
        order = np.argsort(-logits, axis=1, kind="stable")
        ids = experts[order].astype(np.int32)
        sel = np.take_along_axis(logits, order, axis=1)
        return np.ascontiguousarray(ids), _softmax(sel)
    logits = rng.standard_normal((R, E)).astype(np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(logits, order, axis=1)
    return np.ascontiguousarray(order.astype(np.int32)), _softmax(sel)


# ------------------------------------------------------------------ a whole layer

def make_inputs(cfg, R=None, seed=None):
    """Activations and routing (host numpy) for ``cfg``; weights are drawn separately."""
    R = cfg["R"] if R is None else R
    seed = cfg["seed"] if seed is None else seed
    rng = np.random.default_rng([seed, 1])
    z = rng.standard_normal((R, cfg["H"])).astype(np.float32)
    x, sx = activations(z, cfg["kind"])
    ids, w = routing(rng, R, cfg["E"], cfg["k"], cfg["routing"])
    return dict(x=x, sx=sx, ids=ids, w=w, z=z)


def make_layer_numpy(cfg, R=None, seed=None):
    """Everything on the host (small workloads): the dict the oracle's layer functions take."""
    seed = cfg["seed"] if seed is None else seed
    lay = dict(H=cfg["H"], I=cfg["I"], E=cfg["E"], k=cfg["k"], kind=cfg["kind"])
    lay.update(weights_numpy(cfg["E"], cfg["H"], cfg["I"], seed))
    lay.update(make_inputs(cfg, R=R, seed=seed))
    return lay


def plant_nonfinite(lay, row, seed=0):
    """Plant NaN and Inf in one row's activations (bf16: a NaN and a +Inf element; E4M3,
    which has no infinity: the NaN code 0x7F in one element and the NaN scale 0xFF in
    another group)."""
    rng = np.random.default_rng(seed)
    H = lay["H"]
    a, b = rng.choice(H, size=2, replace=False)
    if lay["kind"] == ACT_BF16:
        lay["x"][row, a] = 0x7FC0
        lay["x"][row, b] = 0x7F80
    else:
        lay["x"][row, a] = 0x7F
        g = (b // 32 + 1) % (H // 32) if b // 32 == a // 32 else b // 32
        lay["sx"][row, g] = 0xFF
    return lay
