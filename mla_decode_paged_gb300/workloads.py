"""Seeded synthetic inputs for the MLA paged decode step.

This module only draws random inputs; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle may consume what it
makes.  Every workload's seed is its index (0 for the tiny case, ... 4 for
the ragged batch): the context lengths come from a CPU ``torch.Generator``
seeded with it, and every tensor from a ``torch.Generator`` seeded with it
on the device asked for (CPU for the small cases the oracle
checks in full, the GPU for the full-size cases, where drawing billions of
normals on the host would take minutes).

Workload shapes follow the decode path of the vLLM API page
``vllm.models.kimi_k3.amd.specialized_decode.runtime.mla`` (``m1c_inputs``:
query ``[S, 12, 576]`` bf16, flat fp8 token rows, ``paged_kv_indices`` /
``paged_kv_indptr``, ``scale`` / ``kv_scale``; ``attend``: the padded query
whose row stride spans the pad) and of
``vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value``
(``MlaValue``: W_UV ``[H, 128, 512]`` stored latent-innermost, the gate
``[B, H*128]``, rows ``q`` per request, ``lengths`` per request).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D_QK = 576      # 512 latent ("nope") + 64 rope dims per query / KV row
D_LATENT = 512  # latent width (the value part of a KV row)
D_ROPE = 64
D_V = 128       # W_UV output width per head


@dataclass(frozen=True)
class WorkloadSpec:
    """One synthetic decode workload (sizes, distributions, seed)."""

    name: str
    seed: int
    requests: int
    qlen: int
    heads: int
    heads_pad: int
    lengths: str            # "fixed:a,b,..", "uniform:lo,hi", "const:n", "loguniform:lo,hi"
    kv_scale: float
    zero_requests: int = 0  # requests forced to length 0 (their gate rows NaN)
    pool: str = "sum"       # "sum" (pool = total length) or "rows:N" (pool of N rows)
    scale: float = 1.0 / math.sqrt(192.0)
    splits: tuple = ()      # split counts the workload names (empty: chosen by the plan)
    notes: str = ""

    @property
    def rows(self) -> int:
        return self.requests * self.qlen


# The five workloads: tiny, single-token batch 64, speculative qlen 4,
# long-context 96 heads padded to 128, ragged qlen 8 with empty requests.
WORKLOADS = [
    WorkloadSpec("tiny_r2_h12", 0, 2, 1, 12, 12, "fixed:64,100", 1.0,
                 pool="rows:256", splits=(1, 4),
                 notes="pages = first 164 of a permutation of a 256-row pool"),
    WorkloadSpec("decode_r64_h12", 1, 64, 1, 12, 12, "uniform:1024,8192", 0.8),
    WorkloadSpec("spec_r128_q4_h12", 2, 128, 4, 12, 12, "uniform:4096,32768", 0.8,
                 splits=(8, 32)),
    WorkloadSpec("long_r32_h96p128", 3, 32, 1, 96, 128, "const:32768", 0.8),
    WorkloadSpec("ragged_r256_q8_h12", 4, 256, 8, 12, 12, "loguniform:128,131072",
                 1.25, zero_requests=8),
]


def draw_lengths(spec: WorkloadSpec) -> torch.Tensor:
    """Per-request context lengths (int64, CPU), drawn from the spec's seed."""
    g = torch.Generator().manual_seed(spec.seed)
    kind, _, arg = spec.lengths.partition(":")
    if kind == "fixed":
        lens = torch.tensor([int(x) for x in arg.split(",")], dtype=torch.int64)
    elif kind == "uniform":
        lo, hi = (int(x) for x in arg.split(","))
        lens = torch.randint(lo, hi + 1, (spec.requests,), generator=g)
    elif kind == "const":
        lens = torch.full((spec.requests,), int(arg), dtype=torch.int64)
    elif kind == "loguniform":
        lo, hi = (float(x) for x in arg.split(","))
        u = torch.rand(spec.requests, generator=g, dtype=torch.float64)
        lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
        lens = lens.to(torch.int64).clamp_(int(lo), int(hi))
    else:
        raise ValueError(spec.lengths)
    if spec.zero_requests:
        idx = torch.randperm(spec.requests, generator=g)[: spec.zero_requests]
        lens[idx] = 0
    assert lens.numel() == spec.requests
    return lens


@dataclass
class Inputs:
    """Device tensors of one decode step plus its scalars."""

    spec: WorkloadSpec
    q: torch.Tensor          # bf16 [S, heads_pad, 576] (pad heads NaN)
    kv: torch.Tensor         # uint8 [pool_rows, 576] (fp8 e4m3fn codes)
    pages: torch.Tensor      # int32 [sum L]
    indptr: torch.Tensor     # int32 [R + 1]
    lengths: torch.Tensor    # int32 [R]
    w_uv: torch.Tensor       # bf16 [H, 128, 512]
    gate: torch.Tensor       # bf16 [S, H * 128] raw logits (NaN rows for empty requests)
    scale: float
    kv_scale: float
    extra: dict = field(default_factory=dict)

    @property
    def heads(self) -> int:
        return self.spec.heads

    @property
    def qlen(self) -> int:
        return self.spec.qlen

    @property
    def max_len(self) -> int:
        return int(self.lengths.max().item()) if self.lengths.numel() else 0

    @property
    def total_len(self) -> int:
        return int(self.indptr[-1].item())


def _randn_fp8_codes(rows: int, g: torch.Generator, device, std: float) -> torch.Tensor:
    """[rows, 576] fp8-e4m3fn codes of N(0, std^2) draws, in bounded chunks."""
    out = torch.empty((rows, D_QK), dtype=torch.uint8, device=device)
    step = max(1, (1 << 26) // D_QK)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0, D_QK), generator=g, device=device, dtype=torch.float32)
        out[r0:r1] = (x * std).to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def make_inputs(spec: WorkloadSpec | int, device="cpu", lengths=None) -> Inputs:
    """Draw one workload's tensors on ``device``.

    ``lengths`` (optional, per request) replaces the spec's length draw, for
    edge cases (empty batches, a single long request, ...).  Distributions:
    q ~ N(0,1) bf16; KV ~ N(0, 0.5^2) rounded to fp8 e4m3fn; W_UV ~ N(0, 1/512)
    bf16; gate ~ N(0,1) bf16, NaN on rows of empty requests; pad heads NaN.
    """
    if isinstance(spec, int):
        spec = WORKLOADS[spec]
    device = torch.device(device)
    lens = draw_lengths(spec) if lengths is None else torch.as_tensor(lengths, dtype=torch.int64)
    R = int(lens.numel())
    spec_r = spec if R == spec.requests else _with_requests(spec, R)
    S, H, HP = R * spec.qlen, spec.heads, spec.heads_pad
    total = int(lens.sum().item())

    g = torch.Generator(device=device).manual_seed(spec.seed)
    if spec.pool.startswith("rows:"):
        pool = max(int(spec.pool.split(":")[1]), total)
    else:
        pool = max(total, 1)
    perm = torch.randperm(pool, generator=g, device=device)
    pages = perm[:total].to(torch.int32).contiguous()
    indptr = torch.zeros(R + 1, dtype=torch.int64)
    indptr[1:] = torch.cumsum(lens, 0)
    indptr = indptr.to(torch.int32).to(device)

    q = torch.randn((S, HP, D_QK), generator=g, device=device, dtype=torch.float32)
    q = q.to(torch.bfloat16)
    if HP > H:
        q[:, H:, :] = float("nan")
    kv = _randn_fp8_codes(pool, g, device, 0.5)
    w_uv = (torch.randn((H, D_V, D_LATENT), generator=g, device=device, dtype=torch.float32)
            * (1.0 / math.sqrt(512.0))).to(torch.bfloat16)
    gate = torch.randn((S, H * D_V), generator=g, device=device, dtype=torch.float32)
    gate = gate.to(torch.bfloat16)
    lens_dev = lens.to(torch.int32).to(device)
    empty = (lens == 0).nonzero().flatten()
    for r in empty.tolist():
        gate[r * spec.qlen:(r + 1) * spec.qlen] = float("nan")
    return Inputs(spec_r, q, kv, pages, indptr, lens_dev, w_uv, gate,
                  float(spec.scale), float(spec.kv_scale))


def _with_requests(spec: WorkloadSpec, requests: int) -> WorkloadSpec:
    d = dict(spec.__dict__)
    d["requests"] = requests
    return WorkloadSpec(**d)


def make_latent(rows: int, heads: int, seed: int, device="cpu", std: float = 0.05) -> torch.Tensor:
    """A standalone bf16 latent [rows, heads, 512] ~ N(0, std^2), for testing
    the value/gate stage on its own."""
    g = torch.Generator(device=torch.device(device)).manual_seed(7000 + seed)
    x = torch.randn((rows, heads, D_LATENT), generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def make_partials(splits: int, rows: int, heads: int, seed: int, device="cpu",
                  empty_frac: float = 0.25):
    """Standalone split partials for testing the merge on its own: bf16
    o [splits, rows, heads, 512] and f32 lse [splits, rows, heads], with a
    fraction of the (split, row, head) entries marked empty (lse = -inf, o
    NaN) and some rows empty in every split."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(9000 + seed)
    o = torch.randn((splits, rows, heads, D_LATENT), generator=g, device=dev,
                    dtype=torch.float32).to(torch.bfloat16)
    lse = (torch.randn((splits, rows, heads), generator=g, device=dev, dtype=torch.float32)
           * 3.0 + 5.0)
    drop = torch.rand((splits, rows, heads), generator=g, device=dev) < empty_frac
    if rows > 1:
        drop[:, rows // 2, :] = True  # one row with every split empty
    lse[drop] = float("-inf")
    o[drop] = float("nan")
    return o, lse

def make_block_inputs(spec: WorkloadSpec | int, device="cpu", page_size: int = 16, lengths=None) -> Inputs:
    """A workload's tensors with the KV cache in block-table form (vLLM's
    paged layout with ``page_size`` rows per block): the pool holds whole
    blocks, each request owns ceil(L_r / page_size) distinct random blocks,
    ``pages`` lists block indices, ``indptr`` counts blocks and
    ``extra['last_page_len']`` (int32 [R]) is how many rows of each
    request's last block are used (0 for an empty request).
    ``extra['page_size']`` records the block size.  q, W_UV, gate and the
    value distributions are those of :func:`make_inputs`."""
    if isinstance(spec, int):
        spec = WORKLOADS[spec]
    base = make_inputs(spec, "cpu", lengths=lengths)
    lens = base.lengths.to(torch.int64)
    R = int(lens.numel())
    nb = (lens + page_size - 1) // page_size
    total_blocks = int(nb.sum().item())
    g = torch.Generator().manual_seed(2000 + spec.seed)
    pool_blocks = max(total_blocks + 3, 1)
    blocks = torch.randperm(pool_blocks, generator=g)[:total_blocks].to(torch.int32)
    indptr = torch.zeros(R + 1, dtype=torch.int64)
    indptr[1:] = torch.cumsum(nb, 0)
    last = torch.where(nb > 0, lens - (nb - 1) * page_size, torch.zeros_like(lens)).to(torch.int32)
    kv = _randn_fp8_codes(pool_blocks * page_size, g, "cpu", 0.5)
    device = torch.device(device)
    out = Inputs(base.spec, base.q.to(device), kv.to(device), blocks.to(device), indptr.to(torch.int32).to(device),
                 base.lengths.to(device), base.w_uv.to(device), base.gate.to(device), base.scale, base.kv_scale)
    out.extra["page_size"] = page_size
    out.extra["last_page_len"] = last.to(device)
    return out
