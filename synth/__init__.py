"""Seeded synthetic workloads shaped like the pages' serving scenarios.

This module only draws random tensors. It holds none of the method's arithmetic
(no scoring, selection, quantization or attention), so both the CPU oracle and
the CUDA path can consume the same bytes from it.

Workloads (shapes from the serving scenarios the pages evaluate on; the pages'
own datasets -- LongBench, Needle-in-a-Haystack -- are not available, so seeded
synthetic tensors with these shapes and value distributions stand in for them):

  1 toy          1 layer, 4 MHA heads, d=64, batch 1, prompt 512
  2 llama3-8b    32 layers, 32 q / 8 kv heads, d=128, batch 1, prompt 32,768
  3 llama2-13b   40 layers, 40 MHA heads, d=128, batch 4, prompt 32,768 (no eviction)
  4 mistral-7b   32 layers, 32 q / 8 kv heads, d=128, batch 16 x 8,192
  5 long-ctx     32 layers, 32 q / 8 kv heads, d=128, batch 1, prompt 131,072

Value recipe (all bf16 after one round-to-nearest-even from fp32):
  * toy: Q, K, V ~ N(0, 1).
  * others: key channel c of kv head h in layer l has std sigma_c ~ LogNormal(0, s)
    (s = 0.5, or 1.0 for the long-context workload); K = N(0,1) * sigma_c.
    u_h is a seeded unit vector per (layer, kv head); every query of the group
    is z + 2 u_h with z ~ N(0, I). V ~ N(0, 1).
  * attention sinks: keys at positions 0..3 are 4 * rms * u_h with
    rms = sqrt(sum_c sigma_c^2) (the expected key norm).
  * needles (long-context only): 16 seeded positions per (batch, layer, kv head)
    in [4, n - obs_window); key = 4 * rms * normalize(mean observation query of
    the group).
Seeds: K/V/sigma/u of layer l in workload w use 1000*w + l; the observation
queries use 1000*w + l + 500; decode step t of layer l uses
10,000,000 + 1,000,000*w + 10,000*l + t.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Spec", "WORKLOADS", "workload", "layer_inputs", "decode_inputs",
           "decode_inputs_layers", "small_spec"]


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and distribution of one synthetic workload."""
    wid: int                 # workload id (seeds derive from it)
    name: str
    n_layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    prompt_len: int
    obs_window: int          # 0 = no eviction (quantize-only)
    pool_kernel: int
    schedule: str            # "none" | "uniform" | "pyramid"
    avg_budget: int          # tokens per head (ignored for "none")
    pyramid_depth: int
    bits: int
    group_size: int
    window_len: int          # R, the bf16 recent window
    steps: int               # decode steps
    dist: str = "llm"        # "toy" | "llm"
    sigma_logstd: float = 0.5
    sinks: int = 4
    needles: int = 0

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    1: Spec(1, "toy", 1, 1, 4, 4, 64, 512, 16, 7, "uniform", 128, 0, 2, 32, 32, 16,
            dist="toy", sinks=0),
    2: Spec(2, "llama3-8b", 32, 1, 32, 8, 128, 32768, 32, 7, "pyramid", 512, 8, 2, 32,
            128, 256),
    3: Spec(3, "llama2-13b-quant-only", 40, 4, 40, 40, 128, 32768, 0, 7, "none", 0, 0,
            4, 32, 128, 128),
    4: Spec(4, "mistral-7b-batched", 32, 16, 32, 8, 128, 8192, 32, 7, "uniform", 128,
            0, 2, 32, 64, 512),
    5: Spec(5, "long-context", 32, 1, 32, 8, 128, 131072, 64, 7, "pyramid", 1024, 8, 2,
            32, 128, 1024, sigma_logstd=1.0, needles=16),
}


def workload(wid: int) -> Spec:
    return WORKLOADS[wid]


def small_spec(base: int = 2, **over) -> Spec:
    """A reduced copy of a workload (for tests that the oracle must finish in seconds)."""
    return dataclasses.replace(WORKLOADS[base], **over)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _layer_seed(spec: Spec, layer: int) -> int:
    return 1000 * spec.wid + layer


def _decode_seed(spec: Spec, layer: int, step: int) -> int:
    return 10_000_000 + 1_000_000 * spec.wid + 10_000 * layer + step


def _head_params(spec: Spec, layer: int, device):
    """Per (kv head, channel) key std and per kv head unit direction u_h."""
    g = _gen(_layer_seed(spec, layer) + 77_000, device)
    hk, d = spec.n_kv_heads, spec.head_dim
    sigma = torch.exp(spec.sigma_logstd *
                      torch.randn(hk, d, generator=g, device=device, dtype=torch.float32))
    u = torch.randn(hk, d, generator=g, device=device, dtype=torch.float32)
    u = u / u.norm(dim=-1, keepdim=True)
    return sigma, u


def layer_inputs(spec: Spec, layer: int, device="cpu", with_q: bool = True) -> dict:
    """Prompt tensors of one layer.

    Returns bf16 tensors on `device`:
      q_obs [B][Hq][obs_window][d] (queries of the last obs_window prompt positions),
      k, v  [B][Hkv][n][d],
    and the planted positions `sinks` (list) and `needles` ([B][Hkv][m] int64 or None).
    """
    B, Hq, Hk, d, n, a = (spec.batch, spec.n_q_heads, spec.n_kv_heads, spec.head_dim,
                          spec.prompt_len, spec.obs_window)
    gq = spec.gqa
    seed = _layer_seed(spec, layer)
    gk = _gen(seed, device)
    f32 = torch.float32
    out = {"sinks": [], "needles": None}
    if spec.dist == "toy":
        k = torch.randn(B, Hk, n, d, generator=gk, device=device, dtype=f32)
        v = torch.randn(B, Hk, n, d, generator=gk, device=device, dtype=f32)
        if with_q and a > 0:
            gqn = _gen(seed + 500, device)
            q = torch.randn(B, Hq, a, d, generator=gqn, device=device, dtype=f32)
            out["q_obs"] = q.to(torch.bfloat16)
        out["k"] = k.to(torch.bfloat16)
        out["v"] = v.to(torch.bfloat16)
        return out

    sigma, u = _head_params(spec, layer, device)
    k = torch.randn(B, Hk, n, d, generator=gk, device=device, dtype=f32)
    k.mul_(sigma[None, :, None, :])
    v = torch.randn(B, Hk, n, d, generator=gk, device=device, dtype=f32)
    rms = sigma.pow(2).sum(-1).sqrt()                       # [Hk]
    q = None
    if a > 0:
        gqn = _gen(seed + 500, device)
        z = torch.randn(B, Hq, a, d, generator=gqn, device=device, dtype=f32)
        uq = u.repeat_interleave(gq, dim=0)                  # [Hq][d]
        q = z + 2.0 * uq[None, :, None, :]
    if spec.sinks > 0:
        ns = min(spec.sinks, n)
        k[:, :, :ns, :] = (4.0 * rms[:, None] * u)[None, :, None, :]
        out["sinks"] = list(range(ns))
    if spec.needles > 0 and q is not None:
        gn = _gen(seed + 900, device)
        lo, hi = spec.sinks, n - a
        pos = torch.stack([torch.randperm(hi - lo, generator=gn, device=device)[:spec.needles]
                           for _ in range(B * Hk)]).view(B, Hk, spec.needles) + lo
        pos, _ = pos.sort(dim=-1)
        qm = q.view(B, Hk, gq * a, d).mean(dim=2)           # [B][Hk][d]
        qm = qm / qm.norm(dim=-1, keepdim=True)
        key = 4.0 * rms[None, :, None] * qm                  # [B][Hk][d]
        idx = pos[..., None].expand(B, Hk, spec.needles, d)
        k.scatter_(2, idx, key[:, :, None, :].expand(B, Hk, spec.needles, d).contiguous())
        out["needles"] = pos
    out["k"] = k.to(torch.bfloat16)
    out["v"] = v.to(torch.bfloat16)
    if with_q and q is not None:
        out["q_obs"] = q.to(torch.bfloat16)
    return out


def prompt_queries(spec: Spec, layer: int, device="cpu") -> torch.Tensor:
    """Queries of every prompt position, [B][Hq][n][d] bf16: the first n - obs_window
    drawn like the observation queries (seed stream +700), the last obs_window the
    layer's q_obs itself."""
    B, Hq, d, n, a = spec.batch, spec.n_q_heads, spec.head_dim, spec.prompt_len, spec.obs_window
    g = _gen(_layer_seed(spec, layer) + 700, device)
    z = torch.randn(B, Hq, n - a, d, generator=g, device=device, dtype=torch.float32)
    if spec.dist != "toy":
        _, u = _head_params(spec, layer, device)
        z += 2.0 * u.repeat_interleave(spec.gqa, dim=0)[None, :, None, :]
    head = z.to(torch.bfloat16)
    if a == 0:
        return head
    tail = layer_inputs(spec, layer, device=device)["q_obs"]
    return torch.cat([head, tail], dim=2).contiguous()


def decode_inputs(spec: Spec, layer: int, step: int, device="cpu") -> dict:
    """One decode step of one layer: q [B][Hq][d], k_new, v_new [B][Hkv][d] (bf16)."""
    B, Hq, Hk, d = spec.batch, spec.n_q_heads, spec.n_kv_heads, spec.head_dim
    g = _gen(_decode_seed(spec, layer, step), device)
    f32 = torch.float32
    if spec.dist == "toy":
        q = torch.randn(B, Hq, d, generator=g, device=device, dtype=f32)
        kn = torch.randn(B, Hk, d, generator=g, device=device, dtype=f32)
        vn = torch.randn(B, Hk, d, generator=g, device=device, dtype=f32)
    else:
        sigma, u = _head_params(spec, layer, device)
        z = torch.randn(B, Hq, d, generator=g, device=device, dtype=f32)
        q = z + 2.0 * u.repeat_interleave(spec.gqa, dim=0)[None]
        kn = torch.randn(B, Hk, d, generator=g, device=device, dtype=f32) * sigma[None]
        vn = torch.randn(B, Hk, d, generator=g, device=device, dtype=f32)
    return {"q": q.to(torch.bfloat16), "k_new": kn.to(torch.bfloat16),
            "v_new": vn.to(torch.bfloat16)}


def decode_inputs_layers(spec: Spec, step: int, layers, device="cpu") -> dict:
    """decode_inputs stacked over `layers`: q [L'][B][Hq][d], k_new/v_new [L'][B][Hkv][d]."""
    parts = [decode_inputs(spec, l, step, device) for l in layers]
    return {key: torch.stack([p[key] for p in parts]) for key in ("q", "k_new", "v_new")}
