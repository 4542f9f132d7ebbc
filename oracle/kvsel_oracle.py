"""Plain, slow fp64 CPU oracle for query-aware sparse KV-block selection and
sparse decode attention (the SparPR scheme).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
this module. The product path (the CUDA library and its Python binding) never
does, and this module imports nothing from that path.

Sources (page title, section):
  [SparPR]  "SparPR KV cache recovery on a consumer GPU" news article,
            section "Three decisions rather than one compression ratio":
            paragraph "Query-Aware key-block selection" (block summaries,
            the score, Top-k), paragraph "Dynamic budget control" (copy cost,
            recompute cost, keep ratio, Minimum Keep Floor), paragraph
            "On-demand local recomputation with cost-aware fallback" (span
            merge, Dense Fallback Threshold gamma).
  [DKV]     "DKV: Anchor + Low-Rank Differential KV-Cache Compression",
            abstract (flash-style log-sum-exp merge of partial attentions).
  [Offload] "KV cache offloading" wiki article, section "Why the cache leaves
            the GPU" (KV bytes per token and the transfer-time arithmetic),
            section "NOSA" (blocks kept on the GPU and reused across decode
            steps under an eviction policy: ``BlockCache.step``), the Hugging
            Face Transformers paragraph and section "SparDA" (the next layer's
            blocks fetched ahead of its selection: ``BlockCache.prefetch``).

Every floating-point step is fp64 numpy. Inputs are the bf16 bit patterns
(uint16 arrays) the GPU receives; they are widened to fp64 exactly here.

Readings taken where the pages are silent (each is also listed in the design
notes that accompany the repository):
  * A block summary is the mean key over the block's tokens, one vector per KV
    head ([SparPR] "each head's summary" only makes sense per head).
  * The summary is stored in bf16: the fp64 sum over the block's tokens taken
    sequentially in token order starting from +0.0, divided by the token count
    in fp64, then rounded once from fp64 to bf16 (round to nearest, ties to
    even). A partial last block is averaged over its filled tokens.
  * The score carries no 1/sqrt(d) factor (Top-k is invariant to it); every
    query head h is paired with its GQA KV head kv(h) = h // (H_q / H_kv).
  * Top-k takes the k largest scores, ties to the lower block index; the
    selection is returned in ascending block order.
  * Adjacent means block indices that differ by exactly one.
  * The attended tokens of a selected block are its tokens t < T.
  * Budget: see ``budget``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> fp64, written from the IEEE 754 binary16-brain-float format
# (1 sign bit, 8 exponent bits with bias 127, 7 stored fraction bits).
# ---------------------------------------------------------------------------

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
BF16_MIN_NORMAL = 2.0 ** -126
BF16_SUBNORMAL_QUANTUM = 2.0 ** -133


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def rne_bf16_bits(x) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even); return uint16 bits.

    Done directly from fp64: the value is scaled by the bf16 quantum of its
    binade (a power of two, so the scaling is exact), rounded to an integer
    with ties to even, and scaled back. There is no detour through fp32
    rounding, so no double rounding can occur.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    inf = np.isinf(a)
    fin = ~(nan | inf)
    af = np.where(fin, a, 1.0)
    _, e = np.frexp(af)                      # af = f * 2**e, f in [0.5, 1)
    exp_unbiased = e.astype(np.int64) - 1    # floor(log2(af)) for af > 0
    quantum_exp = np.where(af >= BF16_MIN_NORMAL, exp_unbiased - 7, -133)
    n = np.ldexp(af, -quantum_exp)           # exact: power-of-two scaling
    n = np.rint(n)                           # ties to even
    r = np.ldexp(n, quantum_exp)             # exactly a bf16 value (or 2**128)
    r = np.where(fin, r, 0.0)
    overflow = fin & (r > BF16_MAX)
    with np.errstate(over="ignore"):
        rf = r.astype(np.float32)            # exact: r is representable
    mag = (rf.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    mag = np.where(overflow | inf, np.uint16(0x7F80), mag)
    mag = np.where(nan, np.uint16(0x7FC0), mag)
    out[...] = np.where(sign & ~nan, mag | np.uint16(0x8000), mag)
    return out


# ---------------------------------------------------------------------------
# [Offload] "Why the cache leaves the GPU": KV size and transfer time.
# ---------------------------------------------------------------------------

def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Bytes of K and V one cached token occupies: 2 * layers * kv_heads * head_dim * bytes."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def transfer_seconds(nbytes: float, bytes_per_s: float) -> float:
    """Time to move ``nbytes`` over a link of ``bytes_per_s`` (no overlap, no latency)."""
    return nbytes / bytes_per_s


# ---------------------------------------------------------------------------
# [SparPR] "Query-Aware key-block selection": block summaries.
# ---------------------------------------------------------------------------

def n_blocks(T: int, B: int) -> int:
    return (T + B - 1) // B


def block_sums_f64(k_bits: np.ndarray, T: int, B: int) -> tuple[np.ndarray, np.ndarray]:
    """Per-block fp64 sums of the keys and token counts.

    ``k_bits``: uint16 [>=T][H_kv][d], one sequence in token order.
    Returns (sums [N][H_kv][d] fp64, counts [N] int). Each sum starts at +0.0
    and adds the block's tokens one at a time in token order.
    """
    N = n_blocks(T, B)
    K = bf16_bits_to_f64(k_bits[:T])
    H, d = K.shape[1], K.shape[2]
    sums = np.zeros((N, H, d), dtype=np.float64)
    counts = np.zeros(N, dtype=np.int64)
    n_full = T // B
    if n_full:
        Kb = K[: n_full * B].reshape(n_full, B, H, d)
        acc = np.zeros((n_full, H, d), dtype=np.float64)
        for t in range(B):
            acc = acc + Kb[:, t]
        sums[:n_full] = acc
        counts[:n_full] = B
    if N > n_full:
        acc = np.zeros((H, d), dtype=np.float64)
        for t in range(n_full * B, T):
            acc = acc + K[t]
        sums[n_full] = acc
        counts[n_full] = T - n_full * B
    return sums, counts


def block_summaries(k_bits: np.ndarray, T: int, B: int):
    """bf16 block summaries of one sequence: the mean key per block and KV head.

    Returns (summary bits uint16 [N][H_kv][d], unrounded fp64 means [N][H_kv][d],
    fp64 sum of the last block, which is the open block's accumulator).
    """
    sums, counts = block_sums_f64(k_bits, T, B)
    means = sums / counts[:, None, None].astype(np.float64) if len(counts) else sums
    last = sums[-1].copy() if len(counts) else None
    return rne_bf16_bits(means), means, last


def append_token(acc: np.ndarray | None, k_new_bits: np.ndarray, t: int, B: int):
    """Incremental summary update when token ``t`` is appended.

    A token that opens a new block (t % B == 0) restarts the accumulator from
    +0.0. Returns (new fp64 accumulator, bf16 summary bits of block t // B).
    """
    k = bf16_bits_to_f64(k_new_bits)
    if t % B == 0 or acc is None:
        acc = np.zeros_like(k) + k
    else:
        acc = acc + k
    cnt = t % B + 1
    return acc, rne_bf16_bits(acc / float(cnt))


# ---------------------------------------------------------------------------
# [SparPR] "Query-Aware key-block selection": score and Top-k.
# ---------------------------------------------------------------------------

def kv_head_of(H_q: int, H_kv: int) -> np.ndarray:
    """GQA map: query head h reads KV head h // (H_q / H_kv)."""
    assert H_q % H_kv == 0
    return np.arange(H_q) // (H_q // H_kv)


def block_scores(q_bits: np.ndarray, summary: np.ndarray, summary_is_bits: bool = True) -> np.ndarray:
    """score[n] = sum over query heads h of <q_h, s[n, kv(h)]>, in fp64.

    ``q_bits``: uint16 [H_q][d]; ``summary``: [N][H_kv][d] bf16 bits, or fp64
    values when ``summary_is_bits`` is False.
    """
    q = bf16_bits_to_f64(q_bits)
    s = bf16_bits_to_f64(summary) if summary_is_bits else np.asarray(summary, np.float64)
    kv = kv_head_of(q.shape[0], s.shape[1])
    return np.einsum("hc,nhc->n", q, s[:, kv, :])


def topk_blocks(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores (ties: lower index first), ascending."""
    N = len(scores)
    k = max(0, min(int(k), N))
    idx = np.arange(N)
    order = np.lexsort((idx, -np.asarray(scores, dtype=np.float64)))
    return np.sort(order[:k]).astype(np.int64)


def window_select(scores: np.ndarray, k: int, n_sink: int, n_recent: int) -> np.ndarray:
    """Forced window plus Top-k over the remaining blocks, ascending.

    [DKV] attends a dense recency window exactly beside the Top-k blocks. The
    last ``n_recent`` blocks (and, by the same rule at the other end, the
    first ``n_sink``) are taken whatever their score; the k largest scores
    among the blocks in between are added (ties: lower index). With
    n_sink = n_recent = 0 this is ``topk_blocks``.
    """
    N = len(scores)
    lo = min(int(n_sink), N)
    hi = max(lo, N - int(n_recent))
    forced = list(range(0, lo)) + list(range(hi, N))
    picked = [lo + int(i) for i in topk_blocks(np.asarray(scores, dtype=np.float64)[lo:hi], k)]
    return np.array(sorted(forced + picked), dtype=np.int64)


# ---------------------------------------------------------------------------
# [SparPR] "On-demand local recomputation with cost-aware fallback": spans.
# ---------------------------------------------------------------------------

def merge_spans(sel: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Runs of consecutive block indices -> (starts, lengths)."""
    starts, lens = [], []
    for i, b in enumerate(np.asarray(sel, dtype=np.int64).tolist()):
        if i > 0 and b == prev + 1:
            lens[-1] += 1
        else:
            starts.append(b)
            lens.append(1)
        prev = b
    return np.array(starts, dtype=np.int64), np.array(lens, dtype=np.int64)


def dense_fallback(n_spans: int, k: int, N: int, gamma: float, tau_rel: float) -> bool:
    """Dense Fallback Threshold: go dense once sparse recovery is not clearly cheaper.

    Sparse recovery of k blocks in n_spans spans costs n_spans*tau + k*c_blk;
    dense recovery of all N blocks (one span) costs tau + N*c_blk. With costs in
    units of c_blk (tau_rel = tau / c_blk) the rule is
        dense  iff  n_spans*tau_rel + k >= gamma * (tau_rel + N).
    """
    lhs = float(n_spans) * float(tau_rel) + float(k)
    rhs = float(gamma) * (float(tau_rel) + float(N))
    return lhs >= rhs


# ---------------------------------------------------------------------------
# Attention over the selected blocks ([DKV] for the log-sum-exp form).
# ---------------------------------------------------------------------------

def attend(q_bits, k_bits, v_bits, tokens, scale: float):
    """softmax(q_h . K_t * scale) . V_t over ``tokens`` for every query head.

    q: [H_q][d]; K, V: [T][H_kv][d] (bf16 bits). Returns (out [H_q][d] fp64,
    lse [H_q] fp64, natural log). An empty token set gives out = 0, lse = -inf.
    """
    q = bf16_bits_to_f64(q_bits)
    H_q, d = q.shape
    tokens = np.asarray(tokens, dtype=np.int64)
    out = np.zeros((H_q, d), dtype=np.float64)
    lse = np.full(H_q, -np.inf, dtype=np.float64)
    if tokens.size == 0:
        return out, lse
    K = bf16_bits_to_f64(k_bits[tokens])
    V = bf16_bits_to_f64(v_bits[tokens])
    kv = kv_head_of(H_q, K.shape[1])
    for h in range(H_q):
        logits = (K[:, kv[h], :] @ q[h]) * float(scale)
        m = logits.max()
        p = np.exp(logits - m)
        l = p.sum()
        out[h] = (p @ V[:, kv[h], :]) / l
        lse[h] = m + math.log(l)
    return out, lse


def tokens_of_blocks(blocks, T: int, B: int) -> np.ndarray:
    """Token positions t < T covered by the given block indices, in order."""
    blocks = np.asarray(blocks, dtype=np.int64)
    if blocks.size == 0:
        return np.zeros(0, dtype=np.int64)
    t = (blocks[:, None] * B + np.arange(B)[None, :]).reshape(-1)
    return t[t < T]


# ---------------------------------------------------------------------------
# [SparPR] "Dynamic budget control": copy vs recompute cost -> keep ratio.
# ---------------------------------------------------------------------------

@dataclass
class BudgetOut:
    c_copy_s: float
    c_rec_s: float
    r_model: float
    r: float
    k: int
    tau_rel: float
    dense: bool


def budget(block_size: int, kv_heads: int, head_dim: int, elem_bytes: int, hidden: int,
           n_blocks: int, h2d_bytes_per_s: float, recompute_flop_per_s: float,
           kappa: float = 2.0, keep_floor: float = 0.0, gamma: float = 1.0,
           tau_s: float = 0.0, keep_override: float = -1.0) -> BudgetOut:
    """Per-block copy and recompute costs, keep ratio, k and the dense decision.

    c_copy = 2 * S_blk / BW, S_blk = B * H_kv * d * elem_bytes (the factor 2
    covers K and V). c_rec = kappa * B * hidden^2 / F (cost grows with block
    length and the square of the hidden size; kappa flops per multiply-add).
    The cost ratio maps to the keep ratio as r_model = c_rec / c_copy, the
    share of blocks whose copy costs as much as recomputing them all; the keep
    ratio is r = min(1, max(floor, r_src)) with r_src = keep_override when it
    is >= 0, else r_model. k = clamp(floor(r * N + 1/2), 1, N) (0 when N = 0).
    The host-side dense decision assumes a single span (the cheapest sparse
    case); the device refines it with the actual span count.
    """
    s_blk = float(block_size) * kv_heads * head_dim * elem_bytes
    c_copy = 2.0 * s_blk / float(h2d_bytes_per_s)
    c_rec = float(kappa) * float(block_size) * float(hidden) * float(hidden) / float(recompute_flop_per_s)
    r_model = c_rec / c_copy
    r_src = float(keep_override) if keep_override >= 0.0 else r_model
    r = min(1.0, max(float(keep_floor), r_src))
    if n_blocks <= 0:
        k = 0
    else:
        k = int(math.floor(r * n_blocks + 0.5))
        k = max(1, min(n_blocks, k))
    tau_rel = float(tau_s) / c_copy
    dense = dense_fallback(1, k, n_blocks, gamma, tau_rel) if n_blocks > 0 else False
    return BudgetOut(c_copy, c_rec, r_model, r, k, tau_rel, bool(dense))


# ---------------------------------------------------------------------------
# One decode step for one sequence: the whole path in the pages' order.
# ---------------------------------------------------------------------------

@dataclass
class SeqStep:
    scores: np.ndarray
    sel: np.ndarray
    span_start: np.ndarray
    span_len: np.ndarray
    dense: bool
    out: np.ndarray
    lse: np.ndarray


def decode_seq(q_bits, k_bits, v_bits, T: int, B: int, k: int, scale: float,
               gamma: float = 2.0, tau_rel: float = 0.0, summary_bits=None,
               n_sink: int = 0, n_recent: int = 0) -> SeqStep:
    """Summaries -> scores -> Top-k -> spans -> gamma decision -> attention.

    ``gamma`` defaults to 2 (never dense for k <= N) so that callers opt in to
    the fallback explicitly. ``n_sink`` / ``n_recent`` force the first / last
    blocks into the selection (``window_select``).
    """
    N = n_blocks(T, B)
    if summary_bits is None:
        summary_bits, _, _ = block_summaries(k_bits, T, B) if T > 0 else (np.zeros((0,) + k_bits.shape[1:], np.uint16), None, None)
    scores = block_scores(q_bits, summary_bits) if N > 0 else np.zeros(0)
    sel = window_select(scores, k, n_sink, n_recent)
    ss, sl = merge_spans(sel)
    dense = N > 0 and dense_fallback(len(ss), len(sel), N, gamma, tau_rel)
    blocks = np.arange(N) if dense else sel
    out, lse = attend(q_bits, k_bits, v_bits, tokens_of_blocks(blocks, T, B), scale)
    return SeqStep(scores, sel, ss, sl, bool(dense), out, lse)


# ---------------------------------------------------------------------------
# [Offload] "NOSA": selection is local across consecutive decode steps, so
# blocks fetched in one step are kept on the GPU and reused in the next, and
# an eviction policy bounds the blocks fetched from host memory.
# ---------------------------------------------------------------------------

class BlockCache:
    """GPU-resident copies of host-tier blocks of one sequence, ``slots`` of them.

    Readings where the pages are silent:
      * Eviction is least recently selected first: a slot's stamp is the last
        step in which its block was selected (-1 while empty); the victims are
        the slots not selected in this step with the smallest (stamp, slot
        index), so empty slots go first, in slot order.
      * The misses of a step, taken in ascending block order, fill the victims
        in that order.
      * Full blocks never change; the block holding the last token changes as
        tokens are appended, so when it is selected its copy is fetched again
        even on a hit (into the slot it already holds).
      * A prefetch ("KV cache offloading": the Hugging Face Transformers
        paragraph, the next layer's cache fetched ahead of its use; section
        "SparDA", the blocks a layer will select fetched on a dedicated stream
        while the layer before it runs) loads a predicted block list ahead of
        the selection. It selects nothing: a prefetched block keeps the stamp
        -1 until a step selects it, so a wrong prediction is evicted before any
        block that was ever selected.
    """

    def __init__(self, slots: int):
        self.slots = int(slots)
        self.block_in = [-1] * self.slots
        self.last_use = [-1] * self.slots
        self.slot_of: dict[int, int] = {}

    def step(self, sel, step: int, last_block: int):
        """Serve one step's ascending selection; returns (fetch jobs, hits)
        with each job (block, slot): the misses in ascending block order, then
        the refresh of the last block if it was a hit."""
        sel = [int(n) for n in sel]
        assert len(sel) <= self.slots
        hits, misses, refresh = [], [], []
        for n in sel:
            s = self.slot_of.get(n)
            if s is None:
                misses.append(n)
            else:
                hits.append(n)
                self.last_use[s] = step
                if n == last_block:
                    refresh.append((n, s))
        free = [s for s in range(self.slots) if self.last_use[s] != step]
        free.sort(key=lambda s: (self.last_use[s], s))
        jobs = []
        for n, s in zip(misses, free):
            old = self.block_in[s]
            if old >= 0:
                del self.slot_of[old]
            self.block_in[s] = n
            self.slot_of[n] = s
            self.last_use[s] = step
            jobs.append((n, s))
        return jobs + refresh, hits

    def prefetch(self, pred, last_block: int):
        """Load an ascending predicted block list ahead of the step that may
        select it; returns the fetch jobs (block, slot). The predicted blocks
        that are resident stay where they are, stamps unchanged. The others,
        in ascending block order, take the slots that hold no predicted
        block, smallest (stamp, slot) first, and get the stamp -1. The block
        holding the last token is not prefetched: appends change it until a
        step that selects it fetches it."""
        pred = [int(n) for n in pred]
        assert len(pred) <= self.slots
        assert all(a < b for a, b in zip(pred, pred[1:]))
        keep = {self.slot_of[n] for n in pred if n in self.slot_of}
        misses = [n for n in pred if n not in self.slot_of and n != last_block]
        free = [s for s in range(self.slots) if s not in keep]
        free.sort(key=lambda s: (self.last_use[s], s))
        jobs = []
        for n, s in zip(misses, free):
            old = self.block_in[s]
            if old >= 0:
                del self.slot_of[old]
            self.block_in[s] = n
            self.slot_of[n] = s
            self.last_use[s] = -1
            jobs.append((n, s))
        return jobs
