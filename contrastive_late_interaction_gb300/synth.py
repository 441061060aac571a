"""Seeded synthetic inputs for the contrastive scoring path.

This module only *draws* inputs: Gaussian rows, unit normalisation of the
rows, bf16 rounding, bag memberships, edge lists and ragged lengths.  It holds
none of the loss or MaxSim arithmetic, so both the CPU oracle (through the
tests) and the CUDA path (through the tests and the benchmark) draw their
inputs from here and nowhere else.

Random numbers come from one counter-based generator, written out below from
its published definition (SplitMix64, Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014):

    mix(z):  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9
             z ^= z >> 27; z *= 0x94D049BB133111EB
             z ^= z >> 31
    key(seed, stream) = mix(mix(seed + GAMMA) ^ (stream * 0xD1B54A32D192ED03))
    word(seed, stream, k) = mix(key(seed, stream) + (k + 1) * GAMMA)      (mod 2^64)

with GAMMA = 0x9E3779B97F4A7C15.  A uniform on (0, 1] is
((word >> 11) + 1) * 2^-53, a uniform on [0, 1) is (word >> 11) * 2^-53, and a
standard normal is Box-Muller on two consecutive uniforms (2m, 2m+1):
sqrt(-2 ln u1) * cos(2 pi u2).

Every tensor of a workload draws from its own stream id, so adding a tensor
never shifts another one's values.
"""

from __future__ import annotations

import dataclasses

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)

# Stream ids, one per drawn tensor.
STREAM_EMBEDDINGS = 1
STREAM_BAG_SIZES = 2
STREAM_IGNORE = 3
STREAM_QUERY_LENGTHS = 4
STREAM_DOC_LENGTHS = 5
STREAM_QUERY_ROWS = 6
STREAM_DOC_ROWS = 7
STREAM_D_SCORES = 8
STREAM_SIDES = 9
STREAM_WEIGHTS = 10
STREAM_ARGMAX = 11
STREAM_GROUPS = 12
STREAM_NAMED = 13


# Shift counts as one-element arrays: some numpy releases take a slow path for a uint64 array shifted by a
# uint64 scalar (the values are the same either way).
_S11, _S27, _S30, _S31 = (np.full(1, k, dtype=np.uint64) for k in (11, 27, 30, 31))


def _mix(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> _S30)
        z = z * _M1
        z = z ^ (z >> _S27)
        z = z * _M2
        z = z ^ (z >> _S31)
    return z


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = _mix(np.array([np.uint64(seed % 2**64) + GAMMA], dtype=np.uint64))[0]
        return _mix(np.array([a ^ (np.uint64(stream) * _STREAM_MUL)], dtype=np.uint64))[0]


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit words k = start .. start+count-1 of one stream."""
    key = stream_key(seed, stream)
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + k * GAMMA)


def uniform_open0(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniforms on (0, 1]."""
    w = words(seed, stream, start, count)
    return ((w >> _S11).astype(np.float64) + 1.0) * 2.0**-53


def uniform_closed0(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniforms on [0, 1)."""
    w = words(seed, stream, start, count)
    return (w >> _S11).astype(np.float64) * 2.0**-53


def normal(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Standard normals; normal m uses uniforms 2(start+m) and 2(start+m)+1."""
    u = uniform_open0(seed, stream, 2 * start, 2 * count)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def uniform_int(seed: int, stream: int, count: int, lo: int, hi: int, start: int = 0) -> np.ndarray:
    """Integers uniform on {lo, ..., hi} (inclusive)."""
    u = uniform_closed0(seed, stream, start, count)
    return lo + np.floor(u * (hi - lo + 1)).astype(np.int64)


# ---------------------------------------------------------------------------
# bf16
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        r = (u + rounding) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def unit_rows(seed: int, stream: int, rows: int, width: int, chunk_rows: int = 65536):
    """Gaussian rows L2-normalised in float64, returned as (float32 rows, bf16 bits of those rows)."""
    f32 = np.empty((rows, width), dtype=np.float32)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        g = normal(seed, stream, r0 * width, (r1 - r0) * width).reshape(r1 - r0, width)
        g /= np.sqrt(np.sum(g * g, axis=1, keepdims=True))
        f32[r0:r1] = g.astype(np.float32)
    return f32, bf16_bits(f32)


# ---------------------------------------------------------------------------
# bags and edge sets (CSR: uint64 offsets[count+1], uint32 ids ascending per row)
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Edges:
    offsets: np.ndarray            # uint64 [count + 1]
    ids: np.ndarray                # uint32 [offsets[-1]]
    weights: np.ndarray | None = None   # float32 [offsets[-1]] or None (every edge weighs one)

    @property
    def count(self) -> int:
        return len(self.offsets) - 1


def empty_edges(count: int) -> Edges:
    return Edges(np.zeros(count + 1, dtype=np.uint64), np.zeros(0, dtype=np.uint32))


def edges_from_lists(lists) -> Edges:
    lens = np.array([len(x) for x in lists], dtype=np.uint64)
    offsets = np.zeros(len(lists) + 1, dtype=np.uint64)
    offsets[1:] = np.cumsum(lens)
    ids = np.array([j for x in lists for j in sorted(x)], dtype=np.uint32)
    return Edges(offsets, ids)


def bags_fixed(count: int, size: int) -> np.ndarray:
    return np.arange(count, dtype=np.int64) // size


def bags_uniform(seed: int, count: int, lo: int = 1, hi: int = 4) -> np.ndarray:
    """Bag sizes drawn U{lo..hi} in sequence until `count` items are covered; the last bag is cut."""
    sizes = uniform_int(seed, STREAM_BAG_SIZES, count, lo, hi)
    ends = np.cumsum(sizes)
    nbags = int(np.searchsorted(ends, count) + 1)
    bag = np.repeat(np.arange(nbags, dtype=np.int64), sizes[:nbags])
    return bag[:count]


def attract_within_bags(bag: np.ndarray) -> Edges:
    """Ordered pairs (i, j), i != j, of items sharing a bag."""
    count = len(bag)
    order = np.argsort(bag, kind="stable")
    lists = [None] * count
    b_sorted = bag[order]
    starts = np.flatnonzero(np.r_[True, b_sorted[1:] != b_sorted[:-1]])
    ends = np.r_[starts[1:], count]
    for s, e in zip(starts, ends):
        members = np.sort(order[s:e])
        for i in members:
            lists[i] = [int(j) for j in members if j != i]
    return edges_from_lists(lists)


def ignore_bernoulli(seed: int, count: int, p: float, row_chunk: int = 256) -> Edges:
    """Ordered off-diagonal pairs kept independently with probability p, drawn from word i*count+j."""
    offsets = np.zeros(count + 1, dtype=np.uint64)
    ids = []
    for r0 in range(0, count, row_chunk):
        r1 = min(count, r0 + row_chunk)
        u = uniform_closed0(seed, STREAM_IGNORE, r0 * count, (r1 - r0) * count).reshape(r1 - r0, count)
        keep = u < p
        keep[np.arange(r1 - r0), np.arange(r0, r1)] = False
        rr, cc = np.nonzero(keep)
        ids.append(cc.astype(np.uint32))
        offsets[r0 + 1:r1 + 1] = np.cumsum(np.bincount(rr, minlength=r1 - r0)).astype(np.uint64)
        offsets[r0 + 1:r1 + 1] += offsets[r0]
    return Edges(offsets, np.concatenate(ids) if ids else np.zeros(0, np.uint32))


def diagonal_edges(count: int) -> Edges:
    return Edges(np.arange(count + 1, dtype=np.uint64), np.arange(count, dtype=np.uint32))


def ragged_offsets(lengths: np.ndarray) -> np.ndarray:
    off = np.zeros(len(lengths) + 1, dtype=np.uint64)
    off[1:] = np.cumsum(np.asarray(lengths, dtype=np.uint64))
    return off


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class PooledInputs:
    count: int
    width: int
    e_f32: np.ndarray       # float32 [count, width] (unit rows before bf16 rounding)
    e_bf16: np.ndarray      # uint16 bf16 bits [count, width]
    t: float
    b: float
    attract: Edges
    repel: Edges
    ignore: Edges
    negatives_named: bool = False
    ambient_weight: float = 1.0

    @property
    def e_rounded(self) -> np.ndarray:
        """The exact values the GPU sees (bf16), widened to float64."""
        return bf16_to_f32(self.e_bf16).astype(np.float64)


@dataclasses.dataclass
class MaxSimInputs:
    width: int
    q_offsets: np.ndarray   # uint64 [nq + 1]
    q_bf16: np.ndarray      # uint16 [rows_q, width]
    d_offsets: np.ndarray   # uint64 [nd + 1]
    d_bf16: np.ndarray      # uint16 [rows_d, width]
    d_scores: np.ndarray    # float32 [nq, nd] upstream gradient
    mean: bool = False

    @property
    def nq(self) -> int:
        return len(self.q_offsets) - 1

    @property
    def nd(self) -> int:
        return len(self.d_offsets) - 1

    @property
    def q(self) -> np.ndarray:
        return bf16_to_f32(self.q_bf16).astype(np.float64)

    @property
    def d(self) -> np.ndarray:
        return bf16_to_f32(self.d_bf16).astype(np.float64)


def pooled_tiny(seed: int = 0) -> PooledInputs:
    """N=256, D=64, 128 bags of 2, attract within a bag, repel across bags, diagonal skipped, t=10, b=-10."""
    n, w = 256, 64
    f32, bits = unit_rows(seed, STREAM_EMBEDDINGS, n, w)
    return PooledInputs(n, w, f32, bits, 10.0, -10.0, attract_within_bags(bags_fixed(n, 2)),
                        empty_edges(n), empty_edges(n))


def pooled_bags(seed: int, count: int, width: int, ignore_p: float = 0.0,
                bag_size: int | None = None) -> PooledInputs:
    """Unit Gaussian rows; bags of `bag_size` (or U{1..4}); attract within bags; ambient repel;
    an optional Bernoulli(ignore_p) ignore set over ordered off-diagonal pairs; t=10, b=-10."""
    f32, bits = unit_rows(seed, STREAM_EMBEDDINGS, count, width)
    bag = bags_fixed(count, bag_size) if bag_size else bags_uniform(seed, count)
    ign = ignore_bernoulli(seed, count, ignore_p) if ignore_p > 0 else empty_edges(count)
    return PooledInputs(count, width, f32, bits, 10.0, -10.0, attract_within_bags(bag),
                        empty_edges(count), ign)


def pooled_config2(seed: int = 0) -> PooledInputs:
    return pooled_bags(seed, 4096, 512, ignore_p=0.01)


def pooled_config4(seed: int = 0) -> PooledInputs:
    return pooled_bags(seed, 32768, 768, bag_size=4)


def maxsim_random(seed: int, nq: int, nd: int, width: int, q_len: tuple[int, int],
                  d_len: tuple[int, int]) -> MaxSimInputs:
    """Independent unit rows; query and document lengths uniform on the given inclusive ranges;
    upstream gradient N(0, 1)."""
    ql = uniform_int(seed, STREAM_QUERY_LENGTHS, nq, *q_len)
    dl = uniform_int(seed, STREAM_DOC_LENGTHS, nd, *d_len)
    qo, do = ragged_offsets(ql), ragged_offsets(dl)
    _, qb = unit_rows(seed, STREAM_QUERY_ROWS, int(qo[-1]), width)
    _, db = unit_rows(seed, STREAM_DOC_ROWS, int(do[-1]), width)
    ds = normal(seed, STREAM_D_SCORES, 0, nq * nd).reshape(nq, nd).astype(np.float32)
    return MaxSimInputs(width, qo, qb, do, db, ds)


def maxsim_tiny(seed: int = 0) -> MaxSimInputs:
    """16 queries x 16 docs, query length 8, doc length 32, D=64."""
    return maxsim_random(seed, 16, 16, 64, (8, 8), (32, 32))


def maxsim_config3(seed: int = 0) -> MaxSimInputs:
    return maxsim_random(seed, 512, 512, 128, (8, 64), (32, 1024))


@dataclasses.dataclass
class JointInputs:
    pooled: PooledInputs
    maxsim: MaxSimInputs
    sides: np.ndarray        # uint8 per item: 1 query, 2 document, 3 both
    score_attract: Edges     # attract (i, i) over the score matrix
    score_t: float = 1.0
    score_b: float = 0.0


def joint(seed: int = 0, pooled_count: int = 16384, pooled_width: int = 512, items: int = 2048,
          width: int = 128, d_len=(64, 512), q_len=(16, 48)) -> JointInputs:
    """Pooled part as the U{1..4}-bag recipe without ignores; MaxSim over `items` items whose query
    run is a copy of the first U{q_len} rows of the item's own document run; sides uniform over
    {query, document, both}; the score-matrix loss attracts (i, i) at t=1, b=0."""
    pooled = pooled_bags(seed, pooled_count, pooled_width)
    dl = uniform_int(seed, STREAM_DOC_LENGTHS, items, *d_len)
    ql = np.minimum(uniform_int(seed, STREAM_QUERY_LENGTHS, items, *q_len), dl)
    do, qo = ragged_offsets(dl), ragged_offsets(ql)
    _, db = unit_rows(seed, STREAM_DOC_ROWS, int(do[-1]), width)
    qb = np.concatenate([db[int(do[i]):int(do[i]) + int(ql[i])] for i in range(items)], axis=0)
    ds = np.zeros((items, items), dtype=np.float32)   # replaced by the score loss's gradient
    ms = MaxSimInputs(width, qo, qb, do, db, ds)
    sides = uniform_int(seed, STREAM_SIDES, items, 1, 3).astype(np.uint8)
    return JointInputs(pooled, ms, sides, diagonal_edges(items))


def joint_config5(seed: int = 0) -> JointInputs:
    return joint(seed)


def random_argmax(seed: int, mi: MaxSimInputs) -> np.ndarray:
    """A valid doc-major argmax table [nd, rows_q] drawn uniformly inside each document."""
    rows_q = int(mi.q_offsets[-1])
    dl = np.diff(mi.d_offsets.astype(np.int64))
    u = uniform_closed0(seed, STREAM_ARGMAX, 0, mi.nd * rows_q).reshape(mi.nd, rows_q)
    return np.floor(u * dl[:, None]).astype(np.int32)


def named_documents(seed: int, nq: int, nd: int, others: int) -> tuple[Edges, Edges]:
    """Each query i names its own document i % nd (attract) and `others` further documents drawn uniformly
    without replacement (repel).  Returns (attract, repel) as CSR edge sets over the queries."""
    att, rep = [], []
    for q in range(nq):
        own = q % nd
        draw = uniform_int(seed, STREAM_NAMED, others * 4, 0, nd - 1, start=q * others * 4)
        picked = []
        for d in draw.tolist():
            if d != own and d not in picked:
                picked.append(d)
            if len(picked) == others:
                break
        att.append([own])
        rep.append(sorted(picked))
    return edges_from_lists(att), edges_from_lists(rep)


def maxsim_ties(seed: int, regime: str, nq: int = 24, nd: int = 60, width: int = 64,
                q_len: tuple[int, int] = (1, 70), d_len: tuple[int, int] = (1, 300)) -> MaxSimInputs:
    """MaxSim inputs whose every (query row, document) maximum is an exact tie between identical rows.

    Every query row points along feature 0: q = 0.99 e0 + 0.14 n with n a unit vector on features
    1 .. width/2 - 1.  Each document holds one "winner" row W repeated at 2..5 positions (every row, for
    one document in seven; adjacent documents share W in pairs), the rest "background" rows:
      regime "positive": W = 0.5 e0 + ..., background e0-components in [-0.5, 0.1], so the maximum is
                          the winner, between 0.37 and 0.64;
      regime "negative": W = -0.15 e0 + ..., background in [-0.9, -0.5]: every score is negative and the
                          winner, between -0.29 and -0.01, is the maximum;
      regime "zero":     W is zero on features 0 .. width/2 - 1 (orthogonal to every query row, so its
                          score is exactly zero) and the background is as in "negative".
    The remaining components of each row are a unit vector on the other features, scaled to make the row
    unit.  Identical rows give bit-identical scores on both sides, so the maximum is reached at every
    winner position and the argmax is the lowest one."""
    half = width // 2
    ql = uniform_int(seed, STREAM_QUERY_LENGTHS, nq, *q_len)
    dl = uniform_int(seed, STREAM_DOC_LENGTHS, nd, *d_len)
    qo, do = ragged_offsets(ql), ragged_offsets(dl)
    rows_q, rows_d = int(qo[-1]), int(do[-1])
    n = normal(seed, STREAM_QUERY_ROWS, 0, rows_q * (half - 1)).reshape(rows_q, half - 1)
    n /= np.linalg.norm(n, axis=1, keepdims=True)
    q = np.zeros((rows_q, width))
    q[:, 0] = 0.99
    q[:, 1:half] = 0.14 * n
    u = uniform_closed0(seed, STREAM_DOC_ROWS, 0, rows_d + 8 * nd)
    g = normal(seed, STREAM_DOC_ROWS, rows_d + 8 * nd, (rows_d + nd) * width).reshape(rows_d + nd, width)

    def row(sigma, k, zero_half=False):
        v = g[k].copy()
        v[0] = 0.0
        if zero_half:
            v[:half] = 0.0
        v /= np.linalg.norm(v)
        r = np.sqrt(1.0 - sigma * sigma) * v
        r[0] = sigma
        return r

    w_sigma = {"positive": 0.5, "negative": -0.15, "zero": 0.0}[regime]
    bg_lo, bg_hi = (-0.5, 0.1) if regime == "positive" else (-0.9, -0.5)
    d = np.zeros((rows_d, width))
    winners = [row(w_sigma, rows_d + (i // 2), zero_half=regime == "zero") for i in range(nd)]
    for i in range(nd):
        r0, r1 = int(do[i]), int(do[i + 1])
        length = r1 - r0
        for s in range(length):
            d[r0 + s] = row(bg_lo + (bg_hi - bg_lo) * u[r0 + s], r0 + s)
        if i % 7 == 3:
            pos = np.arange(length)
        else:
            k = min(length, 2 + int(u[rows_d + 8 * i] * 4))
            pick = np.floor(u[rows_d + 8 * i + 1:rows_d + 8 * i + 1 + 2 * k] * length).astype(np.int64)
            pos = np.unique(pick)[:k]
            if length > 1 and pos.size < 2:
                pos = np.array([0, length - 1])
        d[r0 + pos] = winners[i]
    qb = bf16_bits(q.astype(np.float32))
    db = bf16_bits(d.astype(np.float32))
    ds = normal(seed, STREAM_D_SCORES, 0, nq * nd).reshape(nq, nd).astype(np.float32)
    return MaxSimInputs(width, qo, qb, do, db, ds)
