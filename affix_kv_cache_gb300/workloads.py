"""Seeded synthetic inputs for the affix-cache attention path.

This module only draws random tensors and lays out KV slots.  It holds none of the
method's arithmetic (no attention, no importance scores, no anchor selection, no map
building): the CUDA path and the CPU oracle both consume exactly the bits it produces.

Workload shapes follow the pages' evaluation setting (Affix Cache for Diffusion Large
Language Models, Sec. 5 "Default Settings" and "Affix Construction"; App. A prompt
layouts): LLaDA-8B / Dream-7B attention shapes, generation length 256, block 32,
anchor ratio 0.2, affix placed as prefix, infix or suffix.  No dataset or weight is
used; every tensor is drawn from a seeded generator.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from dataclasses import dataclass

import torch

SEG_REQ = "req"
SEG_AFFIX = "affix"
SEG_MASK = "mask"


@dataclass(frozen=True)
class Workload:
    """Geometry and value recipe of one synthetic workload.

    ``segments`` lists the logical sequence left to right as (kind, length) pairs;
    exactly one segment is the shared affix F = [l, l+L).  All non-affix positions are
    probe rows; the ``mask`` positions are the initially masked set M_T.
    """

    name: str
    dtype: str                 # "f32" or "bf16": element type of Q/K/V/O
    layers: int                # N
    hq: int                    # query heads
    hkv: int                   # KV heads (hq % hkv == 0)
    d: int                     # head dim
    batch: int                 # requests B
    segments: tuple            # ((kind, length), ...)
    ratio_permille: int        # anchor ratio in 1/1000; K = ceil(ratio * L)
    recompute_points: int      # recompute points per request (gen length / block)
    plant: str = "none"        # "mean" | "aligned" | "prototypes" | "none"
    plant_count: int = 0       # planted affix positions
    plant_scale: float = 0.0   # magnitude of the planted component
    plant_sigma: float = 0.1   # prototype noise std ("prototypes" only)
    n_prototypes: int = 64
    page: int = 0              # KV slot page size; 0 = contiguous regions
    seed: int = 0

    # ---- derived geometry -------------------------------------------------
    @property
    def T(self) -> int:
        return sum(n for _, n in self.segments)

    @property
    def L(self) -> int:
        return sum(n for k, n in self.segments if k == SEG_AFFIX)

    @property
    def l(self) -> int:
        pos = 0
        for k, n in self.segments:
            if k == SEG_AFFIX:
                return pos
            pos += n
        return 0

    @property
    def P(self) -> int:
        return self.T - self.L

    @property
    def m(self) -> int:
        return sum(n for k, n in self.segments if k == SEG_MASK)

    @property
    def K(self) -> int:
        # ceil(ratio * L) in exact integer arithmetic (ratio held in 1/1000)
        return (self.ratio_permille * self.L + 999) // 1000

    @property
    def R(self) -> int:
        return self.K + self.P

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def probe_positions(self) -> list[int]:
        """Logical positions of the P non-affix rows, ascending."""
        out, pos = [], 0
        for k, n in self.segments:
            if k != SEG_AFFIX:
                out.extend(range(pos, pos + n))
            pos += n
        return out

    def masked_rows(self) -> list[int]:
        """Indices (into the probe rows) of the initially masked positions, ascending."""
        rows, idx = [], 0
        for k, n in self.segments:
            if k == SEG_AFFIX:
                continue
            if k == SEG_MASK:
                rows.extend(range(idx, idx + n))
            idx += n
        return rows

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def describe(self) -> dict:
        return {
            "workload": self.name, "dtype": self.dtype, "layers": self.layers,
            "hq": self.hq, "hkv": self.hkv, "d": self.d, "batch": self.batch,
            "T": self.T, "L": self.L, "l": self.l, "P": self.P, "m": self.m,
            "K": self.K, "R": self.R, "recompute_points": self.recompute_points,
        }


# ---- the workload catalogue ------------------------------------------------
TINY_PREFIX_F32 = Workload(
    name="tiny_prefix_f32", dtype="f32", layers=1, hq=2, hkv=2, d=64, batch=1,
    segments=((SEG_AFFIX, 128), (SEG_REQ, 32), (SEG_MASK, 64)),
    ratio_permille=200, recompute_points=1, plant="mean", plant_count=8,
    plant_scale=2.0, page=0)

LLADA_PREFIX = Workload(
    name="llada8b_prefix_L1024_b4_bf16", dtype="bf16", layers=32, hq=32, hkv=32, d=128,
    batch=4, segments=((SEG_AFFIX, 1024), (SEG_REQ, 128), (SEG_MASK, 256)),
    ratio_permille=200, recompute_points=8, plant="aligned", plant_count=51,
    plant_scale=1.5, page=256)

DREAM_INFIX = Workload(
    name="dream7b_infix_gqa_L2048_b16_bf16", dtype="bf16", layers=28, hq=28, hkv=4,
    d=128, batch=16,
    segments=((SEG_REQ, 256), (SEG_AFFIX, 2048), (SEG_REQ, 64), (SEG_MASK, 256)),
    ratio_permille=200, recompute_points=8, plant="aligned", plant_count=61,
    plant_scale=1.5, page=256)

LLADA_PAGED = Workload(
    name="llada8b_paged_L4096_b16_bf16", dtype="bf16", layers=32, hq=32, hkv=32, d=128,
    batch=16, segments=((SEG_AFFIX, 4096), (SEG_REQ, 128), (SEG_MASK, 256)),
    ratio_permille=200, recompute_points=32, plant="none", page=256)

LLADA_SUFFIX = Workload(
    name="llada8b_suffix_L8192_b32_bf16", dtype="bf16", layers=32, hq=32, hkv=32, d=128,
    batch=32, segments=((SEG_REQ, 256), (SEG_MASK, 256), (SEG_AFFIX, 8192)),
    ratio_permille=200, recompute_points=8, plant="prototypes", plant_count=819,
    plant_sigma=0.1, n_prototypes=64, page=256)

CATALOGUE = {w.name: w for w in
             (TINY_PREFIX_F32, LLADA_PREFIX, DREAM_INFIX, LLADA_PAGED, LLADA_SUFFIX)}


# ---- seeded drawing ----------------------------------------------------------
def _seed(*tags) -> int:
    h = hashlib.sha256(repr(tags).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(w: Workload, device, *tags) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(w.seed, w.layers, w.hq, w.hkv, w.d, w.batch, w.segments, *tags))
    return g


def _randn(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def plant_positions(w: Workload) -> torch.Tensor:
    """Seeded affix offsets that carry a planted key (same for every layer/head)."""
    if w.plant == "none" or w.plant_count == 0:
        return torch.zeros(0, dtype=torch.long)
    g = _gen(w, "cpu", "plant-positions")
    return torch.randperm(w.L, generator=g)[: w.plant_count].sort().values


def probe_inputs(w: Workload, layer: int, device="cpu") -> dict:
    """Probe inputs of one layer.

    Returns q [B][P][Hq][d], k_req / v_req [B][P][Hkv][d] (the request's own K/V,
    rows in ascending logical order) and the shared precomputed affix cache
    k_aff / v_aff [L][Hkv][d], all in the workload's element type.
    """
    B, P, L, hq, hkv, d = w.batch, w.P, w.L, w.hq, w.hkv, w.d
    g = _gen(w, device, "probe", layer)
    k_aff = _randn((L, hkv, d), g, device)
    v_aff = _randn((L, hkv, d), g, device)
    q = _randn((B, P, hq, d), g, device)
    k_req = _randn((B, P, hkv, d), g, device)
    v_req = _randn((B, P, hkv, d), g, device)
    if w.plant != "none" and w.plant_count > 0:
        pos = plant_positions(w).to(device)
        grp = hq // hkv
        if w.plant in ("mean", "aligned"):
            rows = torch.tensor(w.masked_rows(), device=device, dtype=torch.long)
            # mean masked query per KV head: over the batch, the masked rows and the
            # query heads of the group
            qm = q.index_select(1, rows).view(B, len(rows), hkv, grp, d)
            qbar = qm.mean(dim=(0, 1, 3))                       # [hkv][d]
            if w.plant == "mean":
                comp = w.plant_scale * qbar
            else:
                comp = w.plant_scale * math.sqrt(d) * qbar / qbar.norm(dim=-1, keepdim=True)
            k_aff[pos] += comp.unsqueeze(0)
        elif w.plant == "prototypes":
            gp = _gen(w, device, "prototypes", layer)
            protos = _randn((hkv, w.n_prototypes, d), gp, device)
            order = torch.randperm(len(pos), generator=_gen(w, "cpu", "proto-order")).to(device)
            cls = torch.empty(len(pos), dtype=torch.long, device=device)
            cls[order] = torch.arange(len(pos), device=device) % w.n_prototypes
            noise = _randn((len(pos), hkv, d), gp, device) * w.plant_sigma
            k_aff[pos] = protos[:, cls, :].permute(1, 0, 2) + noise
        else:
            raise ValueError(w.plant)
    dt = w.torch_dtype
    return {"q": q.to(dt), "k_req": k_req.to(dt), "v_req": v_req.to(dt),
            "k_aff": k_aff.to(dt), "v_aff": v_aff.to(dt)}


def recompute_inputs(w: Workload, layer: int, point: int = 0, device="cpu") -> dict:
    """Fresh rows of one recompute point of one layer.

    q_r [B][R][Hq][d] are the queries of the R recomputed rows; k_new / v_new
    [B][R][Hkv][d] their freshly recomputed K/V, row i belonging to the i-th
    recomputed logical position (ascending order).
    """
    B, R, hq, hkv, d = w.batch, w.R, w.hq, w.hkv, w.d
    g = _gen(w, device, "recompute", layer, point, w.ratio_permille)
    q_r = _randn((B, R, hq, d), g, device)
    k_new = _randn((B, R, hkv, d), g, device)
    v_new = _randn((B, R, hkv, d), g, device)
    dt = w.torch_dtype
    return {"q_r": q_r.to(dt), "k_new": k_new.to(dt), "v_new": v_new.to(dt)}


BLOCK = 32   # block length of the block-wise decode (Sec. 5, default settings)


def decode_block_positions(w: Workload, step: int) -> list[int]:
    """Logical positions of the block decoded at ``step``: the generation (mask) positions
    are decoded left to right in blocks of ``BLOCK``, cycling when ``step`` passes the last."""
    gen, pos = [], 0
    for k, n in w.segments:
        if k == SEG_MASK:
            gen.extend(range(pos, pos + n))
        pos += n
    n_blocks = max(1, -(-len(gen) // BLOCK))
    i = (step % n_blocks) * BLOCK
    return gen[i:i + BLOCK]


def decode_inputs(w: Workload, layer: int, step: int = 0, device="cpu") -> dict:
    """One block-decode step of one layer: q_blk [B][n][Hq][d] the block's queries, k_blk /
    v_blk [B][n][Hkv][d] its freshly computed K/V (n = the block's length)."""
    n = len(decode_block_positions(w, step))
    g = _gen(w, device, "decode", layer, step)
    q = _randn((w.batch, n, w.hq, w.d), g, device)
    k = _randn((w.batch, n, w.hkv, w.d), g, device)
    v = _randn((w.batch, n, w.hkv, w.d), g, device)
    dt = w.torch_dtype
    return {"q_blk": q.to(dt), "k_blk": k.to(dt), "v_blk": v.to(dt)}


def fresh_context(w: Workload, layer: int, device="cpu") -> dict:
    """Freshly recomputed K/V of every logical position of every request.

    k_fresh / v_fresh [B][T][Hkv][d].  Used to state the end-to-end semantics of
    selective recompute (anchor ratio 0 = direct reuse, 1 = full recompute).
    """
    B, T, hkv, d = w.batch, w.T, w.hkv, w.d
    g = _gen(w, device, "fresh", layer)
    k = _randn((B, T, hkv, d), g, device)
    v = _randn((B, T, hkv, d), g, device)
    dt = w.torch_dtype
    return {"k_fresh": k.to(dt), "v_fresh": v.to(dt)}


@dataclass
class SlotLayout:
    shared_slot: torch.Tensor     # [L] int32: physical slot of affix offset j
    private_slots: torch.Tensor   # [B][R] int32: private slots handed to each request
    num_slots: int
    private_begin: int            # first slot of the private region


def slot_layout(w: Workload, device="cpu") -> SlotLayout:
    """Physical KV slots: the shared affix region first, then per-request private pages.

    With ``page`` > 0 both regions are built from pages of ``page`` slots in a seeded
    shuffled order, so logical neighbours are rarely physical neighbours.
    """
    B, L, R, pg = w.batch, w.L, w.R, w.page
    if pg == 0:
        shared = torch.arange(L, dtype=torch.int32)
        private_begin = L
        private = (L + torch.arange(B * R, dtype=torch.int64)).view(B, R).to(torch.int32)
        num_slots = L + B * R
    else:
        g = _gen(w, "cpu", "slots", w.ratio_permille)
        n_sp = -(-L // pg)
        sperm = torch.randperm(n_sp, generator=g)
        j = torch.arange(L)
        shared = (sperm[j // pg] * pg + j % pg).to(torch.int32)
        private_begin = n_sp * pg
        ppr = -(-R // pg)
        pperm = torch.randperm(B * ppr, generator=g).view(B, ppr)
        i = torch.arange(R)
        private = (private_begin + pperm[:, i // pg] * pg + (i % pg)).to(torch.int32)
        num_slots = private_begin + B * ppr * pg
    return SlotLayout(shared.to(device), private.contiguous().to(device), int(num_slots),
                      int(private_begin))
