"""2D mesh, paired-block placement and double-ring step order (integer math).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[G] "Step 1: 2D Process Mesh Coordinator": a global rank splits into
    seq_rank = rank // p_head and head_rank = rank % p_head; ring neighbours
    differ by one in seq_rank, and the neighbour's global rank is
    seq_rank * p_head + head_rank.
[G] "2. Paired-Block Allocation for Causal Load Balancing" and "Step 2:
    Paired-Block Causal Attention Scheduler": the sequence is cut into
    2 * P_seq blocks and ring rank r owns block r and block 2 * P_seq - 1 - r.
[A] abstract: Double-Ring-Attention is named but not defined.  Reading taken:
    cp = inner * outer; ring rank c sits at (outer index c // inner, inner
    index c % inner).  K/V move one hop around the inner ring per step and,
    after each full inner round, one hop around the outer ring; so at step
    t = o * inner + i rank c holds the K/V that started on rank
    ((c // inner - o) mod outer) * inner + ((c % inner - i) mod inner).
    With outer = 1 this is the single ring of [G] "The Communication Overhead
    and Causal Imbalance of Ring Attention" (rank i receives from rank i - 1).
"""
import numpy as np

ZIGZAG = 1
CONTIGUOUS = 0


def mesh_coords(rank, world_size, p_head):
    """Return the coordinator fields of [G] "Step 1" for one global rank."""
    if world_size % p_head:
        raise ValueError("world size must be divisible by p_head")
    p_seq = world_size // p_head
    seq_rank, head_rank = rank // p_head, rank % p_head
    nxt = (seq_rank + 1) % p_seq
    prv = (seq_rank - 1 + p_seq) % p_seq
    return {
        "p_seq": p_seq,
        "seq_rank": seq_rank,
        "head_rank": head_rank,
        "next_seq_rank": nxt,
        "prev_seq_rank": prv,
        "next_global_rank": nxt * p_head + head_rank,
        "prev_global_rank": prv * p_head + head_rank,
    }


def paired_blocks(p_seq, seq_rank):
    """Block indices (A, B) that ring rank ``seq_rank`` owns ([G] section 2)."""
    return seq_rank, 2 * p_seq - 1 - seq_rank


def rank_blocks(cp, c, placement=ZIGZAG):
    """Natural-order block indices owned by ring rank c, in local order."""
    if placement == ZIGZAG:
        return list(paired_blocks(cp, c))
    return [c]


def block_len(seqlen, cp, placement=ZIGZAG):
    nb = 2 * cp if placement == ZIGZAG else cp
    if seqlen % nb:
        raise ValueError("sequence length must divide into the blocks")
    return seqlen // nb


def rank_tokens(seqlen, cp, c, placement=ZIGZAG):
    """Natural token positions of ring rank c's chunk, in its local order."""
    b = block_len(seqlen, cp, placement)
    return np.concatenate([np.arange(blk * b, (blk + 1) * b)
                           for blk in rank_blocks(cp, c, placement)])


def ring_source(c, t, inner, outer):
    """Ring rank whose K/V rank c holds at step t (double-ring reading)."""
    cp = inner * outer
    if not (0 <= c < cp and 0 <= t < cp):
        raise ValueError("rank or step out of range")
    o, i = divmod(t, inner)
    g, l = divmod(c, inner)
    return ((g - o) % outer) * inner + ((l - i) % inner)


def schedule_table(inner, outer):
    """src[t][c] for every step t and ring rank c."""
    cp = inner * outer
    return np.array([[ring_source(c, t, inner, outer) for c in range(cp)]
                     for t in range(cp)], dtype=np.int64)


def head_group(h, hq, hkv, hp):
    """Query heads and kv heads owned by head rank h (contiguous split).

    [G] "The Scalability Limits of DeepSpeed Ulysses": every head rank keeps
    at least one whole kv head, so hp <= Hkv; [G] "Best Practices", item 2:
    with hp = Hkv each rank has one kv head and Hq / Hkv query heads.
    """
    if hq % hp or hkv % hp or hq % hkv:
        raise ValueError("heads must split evenly over hp")
    nq, nk = hq // hp, hkv // hp
    return list(range(h * nq, (h + 1) * nq)), list(range(h * nk, (h + 1) * nk))


def pair_work(seqlen, cp, c, placement=ZIGZAG):
    """Unmasked (query, key) pairs that ring rank c computes over all steps."""
    qpos = rank_tokens(seqlen, cp, c, placement)
    return int(np.sum(qpos + 1))
