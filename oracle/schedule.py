"""Split-KV schedule: restated rule and the invariants of any valid schedule.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages say only what the schedule is for: FlashMLA computes, ahead of the
kernel and from the sequence lengths alone, which KV segments each SM works on
("get_mla_metadata"), and long contexts at small batch are split along the KV
axis across SMs with the partial results merged afterwards ("MLA 推理：两条计算
路径与 FlashMLA", section "decode 注意力变成了计算问题").  Which rule balances
the work is left open, so any schedule is correct that covers every page of
every request exactly once; ``check_schedule`` tests exactly that.  The library
uses one particular greedy rule, restated in ``schedule_reference`` so that its
integer output can be compared bit for bit:

  nb[b]   = ceil(seqlen[b] / 64)          (0 for an empty request)
  P_eff   = min(P, hbm_parts)             parts that already saturate HBM
  cost    = sum_b nb[b] + F * (#{b : nb[b] > 0} + P_eff - 1)
            (F = cost of one segment in pages; a schedule over P_eff parts has
            at most one segment per request plus one per part boundary)
  target  = ceil(cost / P_eff)
  Parts p = 0..P-1 walk the requests in order.  A part takes whole requests
  while (pages left in it + F) fits in its budget; otherwise it takes
  (budget - F) pages of the current request (at least one) and stops.  The
  last part takes everything still left.  Parts that get nothing are empty.

Metadata row of part p (all int32): [b_first, k_first, b_last, k_end, split_first]
  - empty part: b_first = -1 (the rest 0);
  - otherwise pages [k_first, nb) of b_first, every page of requests strictly
    between, pages [0, k_end) of b_last (or [k_first, k_end) if b_first == b_last);
  - split_first: index, among the segments of request b_first, of the first
    segment of this part (later requests in the part start at segment 0).
num_splits: [B + 1] prefix sums of segments per request.
"""
from __future__ import annotations

PAGE = 64


def pages_of(seqlen: int) -> int:
    return (int(seqlen) + PAGE - 1) // PAGE if seqlen > 0 else 0


def schedule_reference(seqlens, num_parts: int, fixed_cost: int, hbm_parts: int):
    """The greedy rule above.  Returns (meta: list of 5-tuples, num_splits: list)."""
    B = len(seqlens)
    nb = [pages_of(L) for L in seqlens]
    nonempty = sum(1 for n in nb if n > 0)
    p_eff = max(1, min(num_parts, hbm_parts))
    cost = sum(nb) + fixed_cost * (nonempty + p_eff - 1)
    target = (cost + p_eff - 1) // p_eff
    segs = [0] * B
    meta = []
    b, k = 0, 0
    for p in range(num_parts):
        while b < B and nb[b] == 0:
            b += 1
        if b >= B:
            meta.append((-1, 0, 0, 0, 0))
            continue
        first = (b, k, segs[b])
        last_b, last_end = b, k
        budget = target
        while b < B:
            if nb[b] == 0:
                b += 1
                continue
            left = nb[b] - k
            if p == num_parts - 1 or left + fixed_cost <= budget:
                budget -= left + fixed_cost
                segs[b] += 1
                last_b, last_end = b, nb[b]
                b, k = b + 1, 0
            else:
                take = budget - fixed_cost
                if take < 1:
                    break
                k += take
                segs[b] += 1
                last_b, last_end = b, k
                break
        meta.append((first[0], first[1], last_b, last_end, first[2]))
    num_splits = [0] * (B + 1)
    for i in range(B):
        num_splits[i + 1] = num_splits[i] + segs[i]
    return meta, num_splits


def expand_segments(meta, seqlens):
    """List every (part, b, k_begin, k_end, split_index) segment a metadata table describes."""
    nb = [pages_of(L) for L in seqlens]
    out = []
    for p, (b0, k0, b1, k1, s0) in enumerate(meta):
        if b0 < 0:
            continue
        for b in range(b0, b1 + 1):
            if nb[b] == 0:
                continue
            kb = k0 if b == b0 else 0
            ke = k1 if b == b1 else nb[b]
            if ke <= kb:
                continue
            out.append((p, b, kb, ke, s0 if b == b0 else 0))
    return out


def check_schedule(meta, num_splits, seqlens):
    """Invariants of any valid schedule; raises AssertionError with the reason.

    * every page of every request is covered exactly once, by contiguous segments;
    * a request's segments carry split indices 0..n-1 in KV order, and n equals
      num_splits[b+1] - num_splits[b]; empty requests have no segment;
    * within a part, segments follow the global (request, page) order.
    """
    B = len(seqlens)
    nb = [pages_of(L) for L in seqlens]
    segs = expand_segments(meta, seqlens)
    per_req = {b: [] for b in range(B)}
    for p, b, kb, ke, j in segs:
        per_req[b].append((kb, ke, j, p))
    assert num_splits[0] == 0 and len(num_splits) == B + 1
    for b in range(B):
        lst = sorted(per_req[b])
        n = num_splits[b + 1] - num_splits[b]
        assert n == len(lst), f"request {b}: {len(lst)} segments but num_splits says {n}"
        if nb[b] == 0:
            assert not lst, f"empty request {b} has segments"
            continue
        pos = 0
        for idx, (kb, ke, j, _p) in enumerate(lst):
            assert kb == pos, f"request {b}: gap or overlap at page {pos} (segment starts at {kb})"
            assert j == idx, f"request {b}: segment {idx} carries split index {j}"
            pos = ke
        assert pos == nb[b], f"request {b}: covered {pos} of {nb[b]} pages"
    last_key = {}
    for p, b, kb, _ke, _j in segs:
        key = (b, kb)
        if p in last_key:
            assert key > last_key[p], f"part {p}: segments out of order"
        last_key[p] = key
    return True
