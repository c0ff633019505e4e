"""Seeded synthetic inputs for MXFP8 grouped-matmul-finalize-routing.

This module only draws random inputs.  It holds none of the operator's
arithmetic, so the oracle and the CUDA path can both be fed from it without
sharing any part of the computation.

Tensor roles and shapes follow the operator's input table ("MXFP8 实现与精度验证"
write-up, section 3.1, and the aclnnGroupedMatmulFinalizeRoutingV3 parameter
constraints):

    x1              [M, K]                 FP8 bytes (E4M3FN or E5M2), routed tokens
    x2              [E, K, N] or [E, N, K] FP8 bytes, expert weights (transpose_x2)
    scale           [ceil(K/64), N, 2] or [N, ceil(K/64), 2] E8M0 bytes
                    (optionally with a leading E dimension, one slice per expert)
    pertoken_scale  [M, ceil(K/64), 2]     E8M0 bytes
    group_list      [E] int64              prefix sums (type 0) or counts (type 1)
    logit           [M] float32
    row_index       [M] int64              values in [0, batch)
    shared_input    [rows, N] bfloat16
    out             [batch, N] float32     initial value, accumulated into

The input construction mirrors the write-up's test builder (section 3.3:
randn cast to FP8, scales stored as E8M0 bytes, row_index = arange(M) % batch,
bf16 shared input, FP32 zeros for out) and the five workload recipes that the
benchmark and the parity tests use.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

E4M3 = 0
E5M2 = 1
E2M1 = 2  # OCP FP4, two codes per byte along the contiguous dimension, even element in the low nibble

_TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


@dataclasses.dataclass
class Spec:
    """One problem: sizes, formats and the recipe for its random inputs."""

    name: str
    batch: int
    M: int
    K: int
    N: int
    E: int
    x1_dtype: int = E4M3
    x2_dtype: int = E4M3
    transpose_x2: bool = False
    scale_per_expert: bool = False
    group_list_type: int = 1
    # token distribution over experts: "uniform" (equal counts, remainder on
    # the leading experts), "multinomial" (uniform probabilities), "zipf"
    # (probabilities proportional to (i+1)^-zipf_s), or "explicit"
    counts: str = "uniform"
    zipf_s: float = 1.2
    explicit_counts: Optional[tuple] = None
    scale_lo: int = 124
    scale_hi: int = 130
    # row_index recipe: "mod" (arange % batch), "random" (uniform in [0,batch)),
    # "topk" (t // topk)
    rows: str = "mod"
    topk: int = 1
    # logit recipe: "uniform" U(0,1), "softmax" (softmax of topk normals per row), "none"
    logit: str = "uniform"
    shared_rows: Optional[int] = None  # None -> batch; 0 -> no shared input
    shared_offset: int = 0
    shared_weight: float = 1.0
    out_init: str = "zeros"  # "zeros" | "randn"
    bias: bool = False       # per-expert, per-column bf16 bias [E, N] (randn)
    seed: int = 0

    @property
    def Ks(self) -> int:
        return (self.K + 63) // 64

    @property
    def n_shared(self) -> int:
        return self.batch if self.shared_rows is None else self.shared_rows


def _gen(device: str, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def expert_counts(spec: Spec) -> torch.Tensor:
    """Tokens per expert (int64 [E]) for the spec's routing recipe."""
    E, M = spec.E, spec.M
    if spec.counts == "explicit":
        c = torch.tensor(spec.explicit_counts, dtype=torch.int64)
        assert c.numel() == E
        return c
    if spec.counts == "uniform":
        base, rem = divmod(M, E)
        return torch.tensor([base + (1 if i < rem else 0) for i in range(E)], dtype=torch.int64)
    g = _gen("cpu", spec.seed * 7919 + 17)
    if spec.counts == "multinomial":
        p = torch.full((E,), 1.0 / E, dtype=torch.float64)
    elif spec.counts == "zipf":
        p = torch.tensor([(i + 1) ** (-spec.zipf_s) for i in range(E)], dtype=torch.float64)
        p = p / p.sum()
    else:
        raise ValueError(spec.counts)
    draws = torch.multinomial(p, M, replacement=True, generator=g)
    return torch.bincount(draws, minlength=E).to(torch.int64)


def group_list_from_counts(counts: torch.Tensor, group_list_type: int) -> torch.Tensor:
    """Encode per-expert counts as the operator's group_list (type 0 prefix sums, type 1 counts)."""
    if group_list_type == 1:
        return counts.clone()
    if group_list_type == 0:
        return torch.cumsum(counts, 0).to(torch.int64)
    raise ValueError(group_list_type)


def _fp8_bytes(shape, dtype_code: int, g: torch.Generator, device: str) -> torch.Tensor:
    """FP8: randn cast to the format.  E2M1: uniformly random 4-bit codes, two per byte
    along the last dimension (shape is the logical shape; its last size must be even)."""
    if dtype_code == E2M1:
        packed = tuple(shape[:-1]) + (shape[-1] // 2,)
        return torch.randint(0, 256, packed, generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(_TORCH_FP8[dtype_code]).view(torch.uint8)


def _e8m0_bytes(shape, lo: int, hi: int, g: torch.Generator, device: str) -> torch.Tensor:
    return torch.randint(lo, hi + 1, shape, generator=g, device=device, dtype=torch.int32).to(torch.uint8)


def make_inputs(spec: Spec, device: str = "cpu", weights_device: Optional[str] = None) -> Dict[str, torch.Tensor]:
    """Draw every input of one call.  Small tensors are drawn on the CPU from
    fixed seeds; the weight tensor x2 (up to several GB) is drawn on
    ``weights_device`` (default: ``device``) with its own seeded generator."""
    weights_device = weights_device or device
    g = _gen("cpu", spec.seed)
    M, K, N, E, Ks = spec.M, spec.K, spec.N, spec.E, spec.Ks

    x1 = _fp8_bytes((M, K), spec.x1_dtype, g, "cpu")
    gw = _gen(weights_device, spec.seed + 100003)
    wshape = (E, N, K) if spec.transpose_x2 else (E, K, N)
    x2 = _fp8_bytes(wshape, spec.x2_dtype, gw, weights_device)

    sshape = (N, Ks, 2) if spec.transpose_x2 else (Ks, N, 2)
    if spec.scale_per_expert:
        sshape = (E,) + sshape
    scale = _e8m0_bytes(sshape, spec.scale_lo, spec.scale_hi, g, "cpu")
    pertoken_scale = _e8m0_bytes((M, Ks, 2), spec.scale_lo, spec.scale_hi, g, "cpu")

    counts = expert_counts(spec)
    assert int(counts.sum()) <= M
    group_list = group_list_from_counts(counts, spec.group_list_type)

    if spec.logit == "uniform":
        logit = torch.rand((M,), generator=g, dtype=torch.float32)
    elif spec.logit == "softmax":
        z = torch.randn((math.ceil(M / spec.topk), spec.topk), generator=g, dtype=torch.float32)
        logit = torch.softmax(z, dim=1).reshape(-1)[:M].contiguous()
    elif spec.logit == "none":
        logit = None
    else:
        raise ValueError(spec.logit)

    if spec.rows == "mod":
        row_index = torch.arange(M, dtype=torch.int64) % max(spec.batch, 1)
    elif spec.rows == "random":
        row_index = torch.randint(0, spec.batch, (M,), generator=g, dtype=torch.int64)
    elif spec.rows == "topk":
        row_index = torch.arange(M, dtype=torch.int64) // spec.topk
    else:
        raise ValueError(spec.rows)

    R = spec.n_shared
    shared_input = torch.randn((R, N), generator=g, dtype=torch.float32).to(torch.bfloat16) if R > 0 else None

    if spec.out_init == "zeros":
        out = torch.zeros((spec.batch, N), dtype=torch.float32)
    elif spec.out_init == "randn":
        out = torch.randn((spec.batch, N), generator=g, dtype=torch.float32)
    else:
        raise ValueError(spec.out_init)

    bias = torch.randn((E, N), generator=g, dtype=torch.float32).to(torch.bfloat16) if spec.bias else None
    d = dict(x1=x1, x2=x2, scale=scale, pertoken_scale=pertoken_scale, group_list=group_list,
             logit=logit, row_index=row_index, shared_input=shared_input, out=out, bias=bias)
    if device != "cpu":
        d = {k: (v.to(device) if v is not None else None) for k, v in d.items()}
    return d


def _first_seed_with_empty_expert(spec: Spec, start: int) -> int:
    s = start
    while True:
        if int((expert_counts(dataclasses.replace(spec, seed=s)) == 0).sum()) > 0:
            return s
        s += 1


def config(i: int) -> Spec:
    """The five benchmark workloads (1-based), by their sizes and recipes.

    1: batch 64, topk 2, K 5120, N 4096, E 8, E4M3, counts 16/expert (type 1)
    2: batch 128, topk 2, K 7168, N 4096, E 16, E4M3, x2 transposed, shared weight 0.5, out randn
    3: batch 256, topk 3, K 8192, N 4096, E 32, E5M2, prefix sums (type 0), scales 120..134
    4: batch 256, topk 3, K 7168, N 4096, E 32, E4M3, Zipf(1.2) counts, random rows,
       shared 128 rows at offset 64 with weight 0.7
    5: batch 512, topk 8, K 7168, N 4096, E 256, E4M3, multinomial counts, rows t//8,
       softmax logits over the 8 tokens of a row
    """
    if i == 1:
        return Spec("C1 M128 K5120 N4096 E8", batch=64, M=128, K=5120, N=4096, E=8, seed=1001)
    if i == 2:
        return Spec("C2 M256 K7168 N4096 E16 transposed", batch=128, M=256, K=7168, N=4096, E=16,
                    transpose_x2=True, shared_weight=0.5, out_init="randn", seed=1002)
    if i == 3:
        return Spec("C3 M768 K8192 N4096 E32 E5M2", batch=256, M=768, K=8192, N=4096, E=32,
                    x1_dtype=E5M2, x2_dtype=E5M2, group_list_type=0, scale_lo=120, scale_hi=134, seed=1003)
    if i == 4:
        s = Spec("C4 M768 K7168 N4096 E32 zipf", batch=256, M=768, K=7168, N=4096, E=32,
                 counts="zipf", zipf_s=1.2, rows="random", shared_rows=128, shared_offset=64,
                 shared_weight=0.7, seed=1004)
        return dataclasses.replace(s, seed=_first_seed_with_empty_expert(s, 1004))
    if i == 5:
        return Spec("C5 M4096 K7168 N4096 E256", batch=512, M=4096, K=7168, N=4096, E=256,
                    counts="multinomial", rows="topk", topk=8, logit="softmax", seed=1005)
    raise ValueError(i)


def mxfp4_config() -> Spec:
    """The large workload (5) with MXFP4 (E2M1) tokens and weights."""
    return dataclasses.replace(config(5), name="C5-MXFP4 M4096 K7168 N4096 E256", x1_dtype=E2M1, x2_dtype=E2M1,
                               seed=1105)


def mxfp4_small_config() -> Spec:
    """A reduced copy of the MXFP4 large workload (same K, N, tokens per expert and routing
    recipe, 32 experts: 0.5 GB of prepared FP4 weights), sized for full profiler captures."""
    return Spec("MXFP4-E32 M512 K7168 N4096 E32", batch=64, M=512, K=7168, N=4096, E=32, counts="multinomial",
                rows="topk", topk=8, logit="softmax", x1_dtype=E2M1, x2_dtype=E2M1, seed=1106)


def large_small_config() -> Spec:
    """A reduced copy of the large MXFP8 workload (5): the same K, N, tokens per expert and
    routing recipe with 32 experts (about 0.97 GB of prepared weights), sized for full
    profiler captures; its traffic scales to the large workload by the expert count."""
    return Spec("C5-E32 M512 K7168 N4096 E32", batch=64, M=512, K=7168, N=4096, E=32, counts="multinomial",
                rows="topk", topk=8, logit="softmax", seed=1006)


def algorithmic_bytes(spec: Spec, counts: Optional[torch.Tensor] = None) -> int:
    """Bytes a single call must move at minimum: x2 (and its scales) of every
    expert that holds a token, x1, pertoken_scale, logit, row_index,
    group_list, shared_input, the bias rows of those experts, and out read once
    and written once."""
    if counts is None:
        counts = expert_counts(spec)
    nnz = int((counts > 0).sum())
    covered = min(int(counts.sum()), spec.M)
    K, N, Ks = spec.K, spec.N, spec.Ks
    wb = K * N // 2 if spec.x2_dtype == E2M1 else K * N
    w = nnz * wb + nnz * Ks * N * 2 if spec.scale_per_expert else nnz * wb + Ks * N * 2
    tok = covered * (K // 2 if spec.x1_dtype == E2M1 else K) + covered * Ks * 2 + covered * 4 * (0 if spec.logit == "none" else 1) + covered * 8
    shared = spec.n_shared * N * 2
    out = spec.batch * N * 4 * 2
    bias = nnz * N * 2 if spec.bias else 0
    return w + tok + shared + out + spec.E * 8 + bias


def flops(spec: Spec, counts: Optional[torch.Tensor] = None) -> int:
    if counts is None:
        counts = expert_counts(spec)
    return 2 * min(int(counts.sum()), spec.M) * spec.N * spec.K


@dataclasses.dataclass
class RouteSpec:
    """Inputs of the routing step: tokens before routing and a top-k choice of experts."""

    name: str
    batch: int
    topk: int
    K: int
    E: int
    x_dtype: int = E4M3
    invalid: int = 0  # number of (token, k) slots given an expert id outside [0, E)
    seed: int = 0

    @property
    def M(self) -> int:
        return self.batch * self.topk

    @property
    def Ks(self) -> int:
        return (self.K + 63) // 64


def make_route_inputs(spec: RouteSpec) -> Dict[str, torch.Tensor]:
    """topk_ids [batch, topk] int64 (distinct experts per token, uniformly random),
    topk_weights [batch, topk] float32 (softmax of normals), x [batch, K] FP8 bytes,
    x_scale [batch, ceil(K/64), 2] E8M0 bytes in 124..130."""
    g = _gen("cpu", spec.seed)
    scores = torch.rand((spec.batch, spec.E), generator=g)
    ids = torch.topk(scores, k=min(spec.topk, spec.E), dim=1).indices.to(torch.int64)
    if spec.topk > spec.E:
        ids = torch.cat([ids, ids[:, : spec.topk - spec.E]], dim=1)
    if spec.invalid:
        flat = ids.view(-1)
        pos = torch.randperm(flat.numel(), generator=g)[: spec.invalid]
        flat[pos] = torch.where(torch.arange(spec.invalid) % 2 == 0, spec.E + 3, -1)
    w = torch.softmax(torch.randn((spec.batch, spec.topk), generator=g), dim=1)
    x = _fp8_bytes((spec.batch, spec.K), spec.x_dtype, g, "cpu")
    xs = _e8m0_bytes((spec.batch, spec.Ks, 2), 124, 130, g, "cpu")
    return dict(topk_ids=ids.contiguous(), topk_weights=w.contiguous(), x=x, x_scale=xs)


def route_config(i: int) -> RouteSpec:
    """Routing workloads with the batch / topk / K / E of benchmark workloads 1..5."""
    s = config(i)
    return RouteSpec(f"route {s.name.split()[0]} batch{s.batch} topk{s.M // s.batch} K{s.K} E{s.E}",
                     batch=s.batch, topk=s.M // s.batch, K=s.K, E=s.E, x_dtype=s.x1_dtype, seed=2000 + i)


def route_algorithmic_bytes(spec: RouteSpec) -> int:
    """Reads: ids (8 B), weights (4 B), x and x_scale rows once; writes: x1, token
    scales, row_index (8 B), logit (4 B), perm (4 B) per routed entry, group_list."""
    M, K, Ks2 = spec.M, spec.K, 2 * spec.Ks
    return M * 12 + spec.batch * (K + Ks2) + M * (K + Ks2 + 16) + spec.E * 8


@dataclasses.dataclass
class FfnSpec:
    """Grouped SwiGLU expert FFN (BF16): sorted tokens, stacked gate|up and down weights."""

    name: str
    H: int
    I: int
    E: int
    counts: tuple  # tokens per expert
    scale: float = 0.02  # inputs and weights are randn * scale (the write-up's test uses 0.02)
    seed: int = 42


def make_ffn_inputs(spec: FfnSpec, device: str = "cpu", weights_device: Optional[str] = None) -> Dict[str, torch.Tensor]:
    """sorted_tokens [N, H], w13_flat [E*H, 2I], w2_flat [E*I, H] (bf16), expert_cumsum [E+1] int32."""
    weights_device = weights_device or device
    g = _gen("cpu", spec.seed)
    counts = torch.tensor(spec.counts, dtype=torch.int64)
    assert counts.numel() == spec.E
    N = int(counts.sum())
    cs = torch.zeros(spec.E + 1, dtype=torch.int32)
    cs[1:] = torch.cumsum(counts, 0).to(torch.int32)
    x = (torch.randn((N, spec.H), generator=g) * spec.scale).to(torch.bfloat16)
    gw = _gen(weights_device, spec.seed + 7)
    w13 = (torch.randn((spec.E * spec.H, 2 * spec.I), generator=gw, device=weights_device) * spec.scale).to(torch.bfloat16)
    w2 = (torch.randn((spec.E * spec.I, spec.H), generator=gw, device=weights_device) * spec.scale).to(torch.bfloat16)
    d = dict(sorted_tokens=x, w13_flat=w13, w2_flat=w2, expert_cumsum=cs)
    if device != "cpu":
        d = {k: v.to(device) for k, v in d.items()}
    return d


def ffn_config(name: str) -> FfnSpec:
    """'test': the write-up's operator test (H 2048, I 512, counts 0,1,2,4,8,16,32,0);
    'model': LLaDA2.0-mini shape (H 2048, I 512, E 256) with 4096 routed tokens spread
    multinomially over the experts."""
    if name == "test":
        return FfnSpec("ffn test H2048 I512 E8", H=2048, I=512, E=8, counts=(0, 1, 2, 4, 8, 16, 32, 0))
    if name == "model":
        g = _gen("cpu", 4242)
        draws = torch.multinomial(torch.full((256,), 1.0 / 256), 4096, replacement=True, generator=g)
        c = tuple(torch.bincount(draws, minlength=256).tolist())
        return FfnSpec("ffn model H2048 I512 E256 T4096", H=2048, I=512, E=256, counts=c)
    raise ValueError(name)


def ffn_algorithmic_bytes(spec: FfnSpec) -> int:
    """w13 and w2 of experts holding tokens, tokens read, result written (all bf16)."""
    nnz = sum(1 for c in spec.counts if c > 0)
    N = sum(spec.counts)
    return 2 * (nnz * spec.H * 2 * spec.I + nnz * spec.I * spec.H + 2 * N * spec.H) + 4 * (spec.E + 1)


def ffn_flops(spec: FfnSpec) -> int:
    N = sum(spec.counts)
    return 2 * N * spec.H * 2 * spec.I + 2 * N * spec.I * spec.H
