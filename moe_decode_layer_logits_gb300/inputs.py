"""Seeded synthetic inputs for the decode MoE-layer tail.

This module only draws random numbers and stores them in the layouts the
library takes.  It holds none of the method's arithmetic (no GEMM, no top-k,
no softmax, no normalisation), so both the CUDA path and the CPU oracle may be
fed from it.

Value recipe (shapes and distributions of the GLM-5.x decode, MTP-verify and
prefill layer shapes; the second parameter of N(0, s) is a standard
deviation):

* hidden states x and residual ~ N(0, 1) * s, s in {1, 4};
* gate weight W [E, H] ~ N(0, 0.02);
* unfinalized expert rows [N, H] ~ N(0, 0.5), N = T*k rows unless padded;
* expanded-index map [T, k]: a random permutation of the row buffer, or
  (``map_layout="expert_sorted"``) the layout an expert-grouped GEMM writes:
  each token's k slots get k distinct experts drawn uniformly, the (token,
  slot) rows are stored grouped by expert, tokens ascending within a group,
  each group starting on a multiple of ``expert_block`` rows (padding rows
  between groups) when that is > 0;
* shared-expert output ~ N(0, 1);
* gamma = 1 + 0.1 * N(0, 1) in FP32; eps = 1e-6;
* row-parallel partials [R, T, H] ~ N(0, 0.25);
* supplied router logits (prefill) ~ N(0, 0.02 * sqrt(H)) in FP32, the spread
  of x . W at these scales;
* stand-alone routing weights (used when the finalize step is exercised
  without the routing step) ~ U(0, 2 * scale / k) in FP32.

Activations are drawn in float64, narrowed to float32 and then to BF16 with
round-to-nearest-even on the bit pattern.  Every array is reproducible from
(seed, shape, s).
"""

from __future__ import annotations

import numpy as np

__all__ = ["to_bf16_bits", "draw_bf16", "expert_sorted_map", "tail_case", "CONFIGS"]


def to_bf16_bits(a) -> np.ndarray:
    """float64/float32 array -> BF16 bit patterns (uint16) via binary32, RNE."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    out = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    return out


def draw_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape) * std)


def expert_sorted_map(rng: np.random.Generator, T: int, E: int, k: int, block: int = 0):
    """Expert-grouped row layout (see the module docstring).  Returns the map
    [T, k] int32, the number of rows the buffer needs (padding included) and
    the drawn experts [T, k]."""
    experts = np.argsort(rng.random((T, E)), axis=1)[:, :k]  # k distinct experts per token
    e = experts.ravel()
    t = np.repeat(np.arange(T), k)
    order = np.lexsort((t, e))  # by expert, then by token
    counts = np.bincount(e, minlength=E)
    sizes = (counts + block - 1) // block * block if block > 0 else counts
    starts = np.cumsum(sizes) - sizes
    first = np.cumsum(counts) - counts
    se = e[order]
    pos = np.empty(T * k, np.int64)
    pos[order] = starts[se] + (np.arange(T * k) - first[se])
    return pos.reshape(T, k).astype(np.int32), int(sizes.sum()), experts


# Layer shapes of the five workloads: tiny, decode, MTP verify, prefill and
# row-parallel partials.
CONFIGS = {
    "tiny": dict(T=[4], H=[2048], E=64, k=4, scale=1.0, seed=0, R=0),
    "decode": dict(T=[1, 4, 64], H=[6144], E=256, k=8, scale=2.5, seed=1, R=0),
    "verify": dict(T=[4, 12, 28], H=[6144, 2048], E=256, k=8, scale=2.5, seed=2, R=0),
    "prefill": dict(T=[512, 2048, 8192], H=[6144], E=256, k=8, scale=2.5, seed=3, R=0),
    "partials": dict(T=[1, 64, 2048], H=[6144], E=256, k=8, scale=2.5, seed=4, R=4),
}


def tail_case(T: int, H: int, E: int, k: int, *, seed: int, s: float = 1.0,
              scale: float = 2.5, n_rows: int | None = None, shared: bool = True,
              R: int = 0, router: bool = True, logits: bool = False,
              weights: bool = True, eps: float = 1e-6, map_layout: str = "random",
              expert_block: int = 0) -> dict:
    """Draw one layer's inputs.

    Returns a dict of numpy arrays (BF16 as uint16 bit patterns):
    ``x`` [T,H], ``w_gate`` [E,H] (if ``router``), ``rows`` [N,H], ``map``
    [T,k] int32, ``topk_w`` [T,k] float32 (if ``weights``), ``shared`` [T,H]
    or None, ``partials`` [R,T,H] or None, ``residual`` [T,H], ``gamma`` [H]
    float32, ``logits`` [T,E] float32 (if ``logits``), and the scalars.
    """
    rng = np.random.default_rng([int(seed), int(T), int(H), int(E), int(k),
                                 int(round(s * 16)), int(R)])
    if map_layout not in ("random", "expert_sorted"):
        raise ValueError(f"unknown map layout {map_layout!r}")
    sorted_map = map_layout == "expert_sorted" and k > 0
    if sorted_map:
        emap, n_need, _ = expert_sorted_map(rng, T, E, k, expert_block)
    else:
        n_need = T * k
    N = n_need if n_rows is None else int(n_rows)
    if N < n_need:
        raise ValueError("the row buffer must hold at least T*k rows (and the layout's padding)")
    case = dict(T=T, H=H, E=E, k=k, scale=float(scale), eps=float(eps), s=float(s),
                n_rows=N, R=R)
    case["x"] = draw_bf16(rng, (T, H), 1.0 * s)
    case["w_gate"] = draw_bf16(rng, (E, H), 0.02) if router else None
    case["rows"] = draw_bf16(rng, (N, H), 0.5)
    case["map"] = emap if sorted_map else rng.permutation(N)[: T * k].reshape(T, k).astype(np.int32)
    case["shared"] = draw_bf16(rng, (T, H), 1.0) if shared else None
    case["partials"] = draw_bf16(rng, (R, T, H), 0.25) if R > 0 else None
    case["residual"] = draw_bf16(rng, (T, H), 1.0 * s)
    case["gamma"] = (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    if weights:
        hi = 2.0 * scale / max(k, 1)
        case["topk_w"] = rng.uniform(0.0, hi, size=(T, k)).astype(np.float32)
    else:
        case["topk_w"] = None
    if logits:
        case["logits"] = (rng.standard_normal((T, E)) * (0.02 * np.sqrt(H))).astype(np.float32)
    else:
        case["logits"] = None
    return case


def device_layer(T: int, H: int, E: int, k: int, *, seed: int, s: float = 1.0, scale: float = 2.5,
                 shared: bool = True, R: int = 0, router: bool = True, logits: bool = False,
                 map_layout: str = "random", expert_block: int = 0, device="cuda") -> dict:
    """The same recipe drawn directly on the GPU with a seeded torch generator
    (for benchmark buffers too large to draw on the host).  BF16 tensors come
    from FP32 draws rounded to nearest even; output buffers are allocated too.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))

    def bf16(shape, std):
        return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)

    N = T * k
    d = dict(T=T, H=H, E=E, k=k, R=R, scale=float(scale), eps=1e-6)
    d["x"] = bf16((T, H), 1.0 * s) if router else None
    d["w_gate"] = bf16((E, H), 0.02) if router else None
    if map_layout == "expert_sorted" and k > 0:
        # the expert-grouped layout of expert_sorted_map, drawn on the device
        e = torch.rand((T, E), generator=g, device=device).argsort(dim=1)[:, :k].reshape(-1)
        t = torch.arange(T, device=device).repeat_interleave(k)
        order = torch.argsort(e.to(torch.int64) * T + t)
        counts = torch.bincount(e, minlength=E)
        sizes = (counts + expert_block - 1) // expert_block * expert_block if expert_block > 0 else counts
        starts = torch.cumsum(sizes, 0) - sizes
        first = torch.cumsum(counts, 0) - counts
        se = e[order]
        pos = torch.empty(T * k, dtype=torch.int64, device=device)
        pos[order] = starts[se] + (torch.arange(T * k, device=device) - first[se])
        d["map"] = pos.reshape(T, k).to(torch.int32)
        N = int(sizes.sum().item())
        d["rows"] = bf16((max(N, 1), H), 0.5)
    else:
        d["rows"] = bf16((max(N, 1), H), 0.5)
        d["map"] = (torch.randperm(max(N, 1), generator=g, device=device, dtype=torch.int64)[:N]
                    .reshape(T, k).to(torch.int32))
    d["shared"] = bf16((T, H), 1.0) if shared else None
    d["partials"] = bf16((R, T, H), 0.25) if R > 0 else None
    d["residual"] = bf16((T, H), 1.0 * s)
    d["gamma"] = 1.0 + 0.1 * torch.randn(H, generator=g, device=device, dtype=torch.float32)
    d["logits"] = (torch.randn((T, E), generator=g, device=device, dtype=torch.float32) * (0.02 * H ** 0.5)
                   if logits else torch.empty((T, E), device=device, dtype=torch.float32))
    d["topk_ids"] = torch.empty((T, max(k, 1)), device=device, dtype=torch.int32)
    d["topk_w"] = torch.empty((T, max(k, 1)), device=device, dtype=torch.float32)
    d["residual_out"] = torch.empty((T, H), device=device, dtype=torch.bfloat16)
    d["normed_out"] = torch.empty((T, H), device=device, dtype=torch.bfloat16)
    return d
