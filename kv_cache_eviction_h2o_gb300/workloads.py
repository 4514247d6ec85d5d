"""Seeded synthetic workloads for the budgeted-KV decode path.

This module is the one piece shared by the CUDA path's callers and the CPU
oracle's callers: it draws the inputs and nothing else.  It holds none of the
method's arithmetic (no attention, no scores, no eviction, no hashing).

Every array is drawn per (batch*head) unit from ``numpy.random.PCG64`` keyed by
``SeedSequence([seed, tag, unit])``, so any subset of units can be generated
alone and agrees bit for bit with the full tensor.  Half-precision workloads
are rounded to bfloat16 (round to nearest even) here, so the device path and
the oracle read identical values.

Workload shapes follow the model shapes the H2O review page evaluates on
(OPT-6.7B / OPT-30B at a ~20% KV budget, 主な発見 / 提案手法 sections; LLaMA for
long context) with synthetic data in place of model activations.
"""
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

TAG_PROMPT = 1
TAG_DECODE = 2
TAG_SHARED = 3
TAG_LSH = 4
TAG_QUERY = 5          # grouped-query workloads: prompt queries of each query head
TAG_DQUERY = 6         # grouped-query workloads: decode queries of each query head


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    head_dim: int
    prompt: int
    steps: int
    budget: int
    heavy: int
    recent: int
    dtype: str            # "f32" or "bf16"
    seed: int
    structure: tuple = field(default=())
    lsh: bool = False
    lsh_seed: int = 4
    groups: int = 1       # query heads per cache unit (grouped-query attention)
    tau: float = 0.0      # per-head policy workloads: recovery threshold
    full_budget: int = 0  # per-head policy workloads: budget of the full-cache policy

    @property
    def units(self) -> int:
        """Cache units (batch x key/value heads)."""
        return self.batch * self.heads

    @property
    def query_units(self) -> int:
        return self.units * self.groups

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


WORKLOADS = {
    # fp32, 1 x 4 heads, d 64, prompt 128, 64 steps, budget 32 = 16 heavy + 16 recent,
    # rank-2 shared key component of scale 2.
    "tiny": Workload("tiny", 1, 4, 64, 128, 64, 32, 16, 16, "f32", 0, ("rank", 2, 2.0)),
    # OPT-6.7B-shaped layer: 8 x 32 heads, d 128, prompt 2048, 256 steps,
    # budget 410 = 205 heavy + 205 recent, rank-4 shared key component of scale 2.
    "opt-6.7b": Workload("opt-6.7b", 8, 32, 128, 2048, 256, 410, 205, 205, "bf16", 1,
                         ("rank", 4, 2.0)),
    # OPT-30B-shaped layer: 64 x 56 heads, prompt 512, 1024 steps, budget 308 = 154 + 154;
    # 1% of key positions scaled 4x along one shared unit direction.
    "opt-30b": Workload("opt-30b", 64, 56, 128, 512, 1024, 308, 154, 154, "bf16", 2,
                        ("outlier_dir", 0.01, 4.0)),
    # Llama-7B-shaped long context: 1 x 32 heads, prompt 32768, 128 steps,
    # budget 4096 = 2048 + 2048; positions 0..3 and 0.5% of positions get key norm x6.
    "llama-7b-32k": Workload("llama-7b-32k", 1, 32, 128, 32768, 128, 4096, 2048, 2048, "bf16", 3,
                             ("sink_norm", 4, 0.005, 6.0)),
    # HashEvict on the OPT-6.7B shapes and inputs: 32-bit sign projections through a
    # seeded N(0,1) 128 x 32 matrix, recent window 205.
    "hashevict-opt-6.7b": Workload("hashevict-opt-6.7b", 8, 32, 128, 2048, 256, 410, 205, 205,
                                   "bf16", 1, ("rank", 4, 2.0), lsh=True, lsh_seed=4),
    # Per-head policies on the OPT-6.7B shapes: head h of each batch row is a
    # local head (h % 3 == 0), a heavy-hitter head (1) or a broad head (2);
    # recovery threshold 0.95; the full-cache policy keeps prompt + decode.
    "fastgen-opt-6.7b": Workload("fastgen-opt-6.7b", 8, 32, 128, 2048, 256, 410, 205, 205, "bf16", 6,
                                 ("fastgen", 2.0, 0.5, 10.0, 10.0, 0.01, 4, 0.5), tau=0.95, full_budget=2304),
    # The same head mix, small: fp32, head_dim 64, 1 x 6 heads, prompt 256, 32 steps,
    # budget 64 = 32 + 32, full-cache budget 288.
    "fastgen-tiny": Workload("fastgen-tiny", 1, 6, 64, 256, 32, 64, 32, 32, "f32", 7,
                             ("fastgen", 2.0, 0.5, 10.0, 10.0, 0.01, 4, 0.5), tau=0.95, full_budget=288),
    # Grouped-query layer with the OPT-6.7B prompt and budget: 8 x 8 key/value heads,
    # each shared by 4 query heads (32 query heads), d 128, rank-4 keys.
    "gqa-8x8x4": Workload("gqa-8x8x4", 8, 8, 128, 2048, 256, 410, 205, 205, "bf16", 5,
                          ("rank", 4, 2.0), groups=4),
}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); the result
    is float32 holding exactly representable bfloat16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    r = ((u + bias) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32)


def _rng(seed: int, tag: int, index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, index])))


def _shared_direction(w: Workload) -> np.ndarray:
    g = _rng(w.seed, TAG_SHARED, 0)
    u = g.standard_normal(w.head_dim)
    return u / np.linalg.norm(u)


def _unit_basis(w: Workload, unit: int, rank: int) -> np.ndarray:
    g = _rng(w.seed, TAG_SHARED, 1 + unit)
    a = g.standard_normal((w.head_dim, rank))
    qm, _ = np.linalg.qr(a)
    return qm.T.copy()          # [rank, d] orthonormal rows


def _structure_keys(w: Workload, unit: int, K: np.ndarray, g: np.random.Generator,
                    first_pos: int) -> np.ndarray:
    """Apply the workload's key structure to K [n, d] (float64) in place."""
    if not w.structure:
        return K
    kind = w.structure[0]
    n = K.shape[0]
    if kind == "rank":
        rank, amp = int(w.structure[1]), float(w.structure[2])
        basis = _unit_basis(w, unit, rank)
        coef = g.standard_normal((n, rank))
        K += amp * (coef @ basis)
    elif kind == "outlier_dir":
        frac, factor = float(w.structure[1]), float(w.structure[2])
        u = _shared_direction(w)
        mask = g.random(n) < frac
        proj = K[mask] @ u
        K[mask] += (factor - 1.0) * proj[:, None] * u[None, :]
    elif kind == "sink_norm":
        nsink, frac, factor = int(w.structure[1]), float(w.structure[2]), float(w.structure[3])
        mask = g.random(n) < frac
        posn = first_pos + np.arange(n)
        mask |= posn < nsink
        K[mask] *= factor
    else:
        raise ValueError(kind)
    return K


def _finish(w: Workload, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return round_bf16(x) if w.dtype == "bf16" else x


def head_kind(w: Workload, unit: int) -> int:
    """Per-head policy workloads: 0 local head, 1 heavy-hitter head, 2 broad
    head, by the head index of the unit (h % 3)."""
    return (unit % w.heads) % 3


def _positions_embedding(d: int, pos: np.ndarray) -> np.ndarray:
    """[cos(w_m t), sin(w_m t)] over m < d/2, w_m = 10000^(-2m/d): rows whose
    dot product decays with the distance between their positions."""
    m = np.arange(d // 2)
    om = 10000.0 ** (-m / (d // 2))
    t = pos.astype(np.float64)[:, None]
    return np.concatenate([np.cos(om * t), np.sin(om * t)], axis=1)


def _fastgen_qk(w: Workload, unit: int, Q: np.ndarray, K: np.ndarray, g: np.random.Generator,
                first_pos: int):
    """Per-head policy workloads: shape Q, K [n, d] (float64, i.i.d. N(0,1)
    on entry) by the unit's head kind.  Local: amp * E(t) + noise * N for
    both (attention concentrated on nearby positions).  Heavy hitter:
    queries + beta * u, keys N(0,1) with a fraction (and the first nsink
    prompt positions) + gamma * u, u a unit vector of the unit.  Broad:
    scale * N for both (near-uniform attention)."""
    _, amp, noise, beta, gamma, frac, nsink, broad = w.structure
    n, d = Q.shape
    kind = head_kind(w, unit)
    if kind == 0:
        E = _positions_embedding(d, first_pos + np.arange(n))
        return amp * E + noise * Q, amp * E + noise * K
    if kind == 1:
        gu = _rng(w.seed, TAG_SHARED, 1 + unit)
        u = gu.standard_normal(d)
        u /= np.linalg.norm(u)
        mask = g.random(n) < frac
        mask |= (first_pos + np.arange(n)) < nsink
        K = K + np.where(mask[:, None], gamma * u[None, :], 0.0)
        return Q + beta * u[None, :], K
    return broad * Q, broad * K


def prompt_unit(w: Workload, unit: int, prompt: Optional[int] = None):
    """Prompt Q, K, V of one unit, each [T, d] float32."""
    T = w.prompt if prompt is None else prompt
    g = _rng(w.seed, TAG_PROMPT, unit)
    d = w.head_dim
    Q = g.standard_normal((T, d), dtype=np.float32).astype(np.float64)
    K = g.standard_normal((T, d), dtype=np.float32).astype(np.float64)
    V = g.standard_normal((T, d), dtype=np.float32).astype(np.float64)
    if w.structure and w.structure[0] == "fastgen":
        Q, K = _fastgen_qk(w, unit, Q, K, g, 0)
    else:
        K = _structure_keys(w, unit, K, g, 0)
    return _finish(w, Q), _finish(w, K), _finish(w, V)


def decode_unit(w: Workload, unit: int, steps: Optional[int] = None,
                prompt: Optional[int] = None):
    """Decode-step q, k, v of one unit, each [S, d] float32; the new keys get
    the same structure as the prompt keys."""
    S = w.steps if steps is None else steps
    T = w.prompt if prompt is None else prompt
    g = _rng(w.seed, TAG_DECODE, unit)
    d = w.head_dim
    q = g.standard_normal((S, d), dtype=np.float32).astype(np.float64)
    k = g.standard_normal((S, d), dtype=np.float32).astype(np.float64)
    v = g.standard_normal((S, d), dtype=np.float32).astype(np.float64)
    if w.structure and w.structure[0] == "fastgen":
        q, k = _fastgen_qk(w, unit, q, k, g, T)
    else:
        k = _structure_keys(w, unit, k, g, T)
    return _finish(w, q), _finish(w, k), _finish(w, v)


def query_rows(w: Workload, qunit: int, n: int, decode: bool) -> np.ndarray:
    """Grouped-query workloads: prompt (or decode) queries [n, d] of query
    head `qunit` (head g of cache unit u is qunit = u * groups + g)."""
    g = _rng(w.seed, TAG_DQUERY if decode else TAG_QUERY, qunit)
    return _finish(w, g.standard_normal((n, w.head_dim), dtype=np.float32))


def lsh_matrix(w: Workload) -> np.ndarray:
    """HashEvict projection matrix W [d, 32] float32, N(0, 1)."""
    g = _rng(w.lsh_seed, TAG_LSH, 0)
    return g.standard_normal((w.head_dim, 32), dtype=np.float32)


def generate(w: Workload, units: Optional[Sequence[int]] = None,
             steps: Optional[int] = None, prompt: Optional[int] = None):
    """Inputs for the listed (cache) units (default all): dict with Q, K, V
    [U, T, d] and q, k, v [S, U, d] (float32) plus W for LSH workloads.  A
    grouped-query workload has G = groups query heads per unit: Q [U*G, T, d]
    and q [S, U*G, d], head g of the i-th listed unit in row i * G + g."""
    if units is None:
        units = range(w.units)
    units = list(units)
    S = w.steps if steps is None else steps
    T = w.prompt if prompt is None else prompt
    d = w.head_dim
    U, G = len(units), w.groups
    out = {
        "Q": np.empty((U * G, T, d), np.float32), "K": np.empty((U, T, d), np.float32),
        "V": np.empty((U, T, d), np.float32), "q": np.empty((S, U * G, d), np.float32),
        "k": np.empty((S, U, d), np.float32), "v": np.empty((S, U, d), np.float32),
    }
    for i, u in enumerate(units):
        Qu, out["K"][i], out["V"][i] = prompt_unit(w, u, T)
        if S > 0:
            qu, out["k"][:, i], out["v"][:, i] = decode_unit(w, u, S, T)
        if G == 1:
            out["Q"][i] = Qu
            if S > 0:
                out["q"][:, i] = qu
            continue
        for j in range(G):
            out["Q"][i * G + j] = query_rows(w, u * G + j, T, False)
            if S > 0:
                out["q"][:, i * G + j] = query_rows(w, u * G + j, S, True)
    if w.lsh:
        out["W"] = lsh_matrix(w)
    return out


def generate_device(w: Workload, seed_offset: int = 0, prompt: Optional[int] = None,
                    steps: Optional[int] = None, device: str = "cuda"):
    """The same recipe drawn with torch's device generator, for full-size
    benchmark pools (values differ from ``generate``; distributions and
    structure match).  Returns device tensors Q, K, V [U, T, d] and q, k, v
    [S, U, d] in the workload's element type, plus W [d, 32] for LSH; a
    grouped-query workload's Q and q have U * groups rows."""
    import torch

    T = w.prompt if prompt is None else prompt
    S = w.steps if steps is None else steps
    U, d = w.units, w.head_dim
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * (w.seed + 1) + seed_offset)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def normal(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)

    basis = None
    if w.structure and w.structure[0] == "rank":
        rank = int(w.structure[1])
        gb = _rng(w.seed, TAG_SHARED, 1_000_000 + seed_offset)
        qb = np.linalg.qr(gb.standard_normal((U, d, rank)))[0]           # [U, d, rank]
        basis = torch.from_numpy(np.ascontiguousarray(qb.transpose(0, 2, 1), np.float32)).to(device)
    u_dir = None
    if w.structure and w.structure[0] == "outlier_dir":
        u_dir = normal(d)
        u_dir = u_dir / u_dir.norm()

    def keys(Kx, first_pos):
        # Kx: [U, n, d] (prompt) or [n, U, d] transposed by the caller
        if not w.structure:
            return Kx
        kind = w.structure[0]
        n = Kx.shape[1]
        if kind == "rank":
            coef = normal(U, n, basis.shape[1])
            return Kx + float(w.structure[2]) * torch.bmm(coef, basis)
        if kind == "outlier_dir":
            frac, factor = float(w.structure[1]), float(w.structure[2])
            mask = (torch.rand(U, n, generator=g, device=device) < frac).unsqueeze(-1)
            proj = (Kx @ u_dir).unsqueeze(-1) * u_dir
            return torch.where(mask, Kx + (factor - 1.0) * proj, Kx)
        if kind == "sink_norm":
            nsink, frac, factor = int(w.structure[1]), float(w.structure[2]), float(w.structure[3])
            mask = torch.rand(U, n, generator=g, device=device) < frac
            posn = first_pos + torch.arange(n, device=device)
            mask |= (posn < nsink).unsqueeze(0)
            return torch.where(mask.unsqueeze(-1), Kx * factor, Kx)
        raise ValueError(kind)

    if w.structure and w.structure[0] == "fastgen":
        _, amp, noise, beta, gamma, frac, nsink, broad = w.structure
        kind = torch.tensor([head_kind(w, u) for u in range(U)], device=device).view(U, 1, 1)
        udir = normal(U, d)
        udir = (udir / udir.norm(dim=1, keepdim=True)).unsqueeze(1)

        def emb(first, n):
            return torch.from_numpy(_positions_embedding(d, first + np.arange(n)).astype(np.float32)).to(device)

        def fastgen(Qx, Kx, first):
            # Qx, Kx: [U, n, d] N(0,1); the three head kinds as in the numpy recipe
            n = Qx.shape[1]
            E = emb(first, n).unsqueeze(0)
            mask = (torch.rand(U, n, 1, generator=g, device=device) < frac) | \
                ((first + torch.arange(n, device=device)) < nsink).view(1, n, 1)
            Ql, Kl = amp * E + noise * Qx, amp * E + noise * Kx
            Qh, Kh = Qx + beta * udir, Kx + torch.where(mask, gamma * udir, torch.zeros_like(Kx))
            Qb, Kb = broad * Qx, broad * Kx
            Qo = torch.where(kind == 0, Ql, torch.where(kind == 1, Qh, Qb))
            Ko = torch.where(kind == 0, Kl, torch.where(kind == 1, Kh, Kb))
            return Qo, Ko

        Qp, Kp = fastgen(normal(U, T, d), normal(U, T, d), 0)
        out = {"Q": Qp.to(dt).contiguous(), "K": Kp.to(dt).contiguous(), "V": normal(U, T, d).to(dt).contiguous()}
        if S > 0:
            qd, kd = fastgen(normal(U, S, d), normal(U, S, d), T)
            out["q"] = qd.transpose(0, 1).to(dt).contiguous()
            out["k"] = kd.transpose(0, 1).to(dt).contiguous()
            out["v"] = normal(S, U, d).to(dt).contiguous()
        return out

    out = {
        "Q": normal(U * w.groups, T, d).to(dt).contiguous(),
        "K": keys(normal(U, T, d), 0).to(dt).contiguous(),
        "V": normal(U, T, d).to(dt).contiguous(),
    }
    if S > 0:
        out["q"] = normal(S, U * w.groups, d).to(dt).contiguous()
        out["k"] = keys(normal(U, S, d), T).transpose(0, 1).to(dt).contiguous()
        out["v"] = normal(S, U, d).to(dt).contiguous()
    if w.lsh:
        out["W"] = torch.from_numpy(lsh_matrix(w)).to(device)
    return out
