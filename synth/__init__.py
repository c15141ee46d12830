"""Seeded synthetic inputs for the recurrence workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
holds only input generation (shapes and value distributions); none of the
recurrence arithmetic lives here, so neither the CPU oracle nor the GPU
library depends on the other through it.

Every tensor is fp32, contiguous, drawn from a ``torch.Generator`` seeded with
``1000 * config_id + tensor_id``.  The same call with ``device="cpu"`` always
returns the same values on one machine; ``device="cuda"`` draws from the CUDA
generator instead (used by the benchmark, whose inputs only need the right
distribution).

Workload recipes (page sources: "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的
C 推理运行时" §2.2, §4.1-§4.3, §5.1; the value distributions and sizes are the
benchmark configurations this library is measured on):

* scan_small   B=2 T=128 N=128:  a = sigmoid(N(0,1)), b,u ~ N(0,1), s0 = 0.
* scan_large   B=8 T=8192 N=2048: a = sigmoid(N(1.5,1)), b,u ~ N(0,1), s0 ~ N(0,1).
* gla          B=4 T=4096 H=4 dk=dv=128: q,k,v ~ N(0,1)/sqrt(dk),
               d = exp(logsigmoid(N(0,1))/16) per key, scale = dk^-1/2, S0 = 0.
* mamba2       B=4 T=4096 H=24 G=1 dk=128 (state) dv=64 (head dim):
               dt = softplus(N(0,1)) per (b,t,h), A = -exp(U(0,1)) per head,
               dA = exp(dt*A), k = B_g ~ N(0,1), v = dt * x with x ~ N(0,1),
               q = C_g ~ N(0,1), scale = 1, S0 = 0.
* deltanet     B=4 T=4096 H=8 dk=dv=128: k,q = L2-normalised N(0,1), v ~ N(0,1),
               beta = sigmoid(N(0,1)), scale = 1, S0 = 0.
* rwkv7        B=16 T=4096 H=12 dk=dv=64 (prefill, S0 = 0) and B=1024 T=1
               (decode, S0 ~ N(0,1)): w = exp(-exp(N(-0.5,0.5))) per key column,
               k = L2-normalised N(0,1), v,q ~ N(0,1).
"""
from __future__ import annotations

import math

import torch

CONFIGS = {
    "scan_small": dict(cid=1, B=2, T=128, N=128),
    "scan_large": dict(cid=2, B=8, T=8192, N=2048),
    "gla": dict(cid=3, B=4, T=4096, H=4, G=4, dk=128, dv=128),
    "mamba2": dict(cid=4, B=4, T=4096, H=24, G=1, dk=128, dv=64),
    "deltanet": dict(cid=5, B=4, T=4096, H=8, dk=128, dv=128),
    "rwkv7_prefill": dict(cid=6, B=16, T=4096, H=12, dk=64, dv=64),
    "rwkv7_decode": dict(cid=7, B=1024, T=1, H=12, dk=64, dv=64),
    # not a benchmark configuration of the pages: the GLA shape run through the
    # gated (convex-combination) matrix state
    "gated_memory": dict(cid=8, B=4, T=4096, H=4, G=4, dk=128, dv=128),
}

DECAY_PER_KEY = 0
DECAY_PER_HEAD = 1
DECAY_PER_KEY_GATED = 2
DECAY_PER_HEAD_GATED = 3


def _gen(seed: int, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed, mean=0.0, std=1.0, device="cpu"):
    x = torch.empty(shape, dtype=torch.float32, device=device)
    return x.normal_(mean, std, generator=_gen(seed, device))


def uniform(shape, seed, lo=0.0, hi=1.0, device="cpu"):
    x = torch.empty(shape, dtype=torch.float32, device=device)
    return x.uniform_(lo, hi, generator=_gen(seed, device))


def _l2n(x):
    return (x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)).contiguous()


def scan_inputs(B, T, N, *, large=False, cid=None, device="cpu"):
    """Inputs of both scan forms: dict(a, b, u, s0).  ``large`` selects the
    large-workload distribution (decays near 0.8, random s0)."""
    cid = (2 if large else 1) if cid is None else cid
    s = 1000 * cid
    if large:
        a = torch.sigmoid(normal((B, T, N), s + 1, 1.5, 1.0, device))
        s0 = normal((B, N), s + 4, device=device)
    else:
        a = torch.sigmoid(normal((B, T, N), s + 1, device=device))
        s0 = None
    b = normal((B, T, N), s + 2, device=device)
    u = normal((B, T, N), s + 3, device=device)
    return dict(a=a.contiguous(), b=b, u=u, s0=s0)


def gla_inputs(B, T, H, dk, dv, *, cid=3, device="cpu"):
    s = 1000 * cid
    r = 1.0 / math.sqrt(dk)
    q = normal((B, T, H, dk), s + 1, device=device) * r
    k = normal((B, T, H, dk), s + 2, device=device) * r
    v = normal((B, T, H, dv), s + 3, device=device) * r
    gk = torch.nn.functional.logsigmoid(normal((B, T, H, dk), s + 4, device=device)) / 16.0
    d = torch.exp(gk)
    return dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(), d=d.contiguous(),
                S0=None, H=H, G=H, decay_kind=DECAY_PER_KEY, scale=dk ** -0.5)


def mamba2_inputs(B, T, H, G, dk, dv, *, cid=4, device="cpu"):
    s = 1000 * cid
    dt = torch.nn.functional.softplus(normal((B, T, H), s + 1, device=device))
    A = -torch.exp(uniform((H,), s + 2, device=device))
    dA = torch.exp(dt * A)
    k = normal((B, T, G, dk), s + 3, device=device)          # B_g
    x = normal((B, T, H, dv), s + 4, device=device)
    v = dt[..., None] * x                                     # dt folded into the value
    q = normal((B, T, G, dk), s + 5, device=device)          # C_g
    return dict(q=q, k=k, v=v.contiguous(), d=dA.contiguous(), S0=None, H=H, G=G,
                decay_kind=DECAY_PER_HEAD, scale=1.0)


def deltanet_inputs(B, T, H, dk, dv, *, cid=5, device="cpu"):
    s = 1000 * cid
    k = _l2n(normal((B, T, H, dk), s + 1, device=device))
    q = _l2n(normal((B, T, H, dk), s + 2, device=device))
    v = normal((B, T, H, dv), s + 3, device=device)
    beta = torch.sigmoid(normal((B, T, H), s + 4, device=device)).contiguous()
    return dict(q=q, k=k, v=v, beta=beta, S0=None, scale=1.0)


def rwkv7_inputs(B, T, H, dk, dv, *, random_state=False, cid=6, device="cpu"):
    s = 1000 * cid
    w = torch.exp(-torch.exp(normal((B, T, H, dk), s + 1, -0.5, 0.5, device))).contiguous()
    k = _l2n(normal((B, T, H, dk), s + 2, device=device))
    v = normal((B, T, H, dv), s + 3, device=device)
    q = normal((B, T, H, dk), s + 4, device=device)
    S0 = normal((B, H, dv, dk), s + 5, device=device) if random_state else None
    return dict(q=q, k=k, v=v, w=w, S0=S0)


def gated_memory_inputs(B, T, H, dk, dv, *, per_key=True, cid=8, device="cpu"):
    """Gated matrix state S = p (.) S + (1 - p) (.) (k v^T): the GLA-shaped
    inputs with the gate p = sigmoid(N(2,1)) (mostly retaining), per key or
    per head, scale dk^-1/2."""
    s = 1000 * cid
    r = 1.0 / math.sqrt(dk)
    q = normal((B, T, H, dk), s + 1, device=device) * r
    k = normal((B, T, H, dk), s + 2, device=device) * r
    v = normal((B, T, H, dv), s + 3, device=device)
    shape = (B, T, H, dk) if per_key else (B, T, H)
    p = torch.sigmoid(normal(shape, s + 4, 2.0, 1.0, device))
    return dict(q=q.contiguous(), k=k.contiguous(), v=v, d=p.contiguous(), S0=None, H=H, G=H,
                decay_kind=DECAY_PER_KEY_GATED if per_key else DECAY_PER_HEAD_GATED, scale=dk ** -0.5)


def config_inputs(name, device="cpu", **override):
    """Inputs of a named workload, with optional shape overrides."""
    c = dict(CONFIGS[name])
    c.update(override)
    cid = c.pop("cid")
    if name.startswith("scan"):
        return scan_inputs(c["B"], c["T"], c["N"], large=(name == "scan_large"), cid=cid, device=device)
    if name == "gla":
        return gla_inputs(c["B"], c["T"], c["H"], c["dk"], c["dv"], cid=cid, device=device)
    if name == "mamba2":
        return mamba2_inputs(c["B"], c["T"], c["H"], c["G"], c["dk"], c["dv"], cid=cid, device=device)
    if name == "deltanet":
        return deltanet_inputs(c["B"], c["T"], c["H"], c["dk"], c["dv"], cid=cid, device=device)
    if name == "gated_memory":
        return gated_memory_inputs(c["B"], c["T"], c["H"], c["dk"], c["dv"], cid=cid, device=device)
    if name.startswith("rwkv7"):
        return rwkv7_inputs(c["B"], c["T"], c["H"], c["dk"], c["dv"],
                            random_state=(name == "rwkv7_decode"), cid=cid, device=device)
    raise KeyError(name)
