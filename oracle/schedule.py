"""Split-KV schedule: restated rule and the invariants of any valid schedule.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages say only what the schedule is for: FlashMLA computes, ahead of the
kernel and from the sequence lengths alone, which KV segments each SM works on
("get_mla_metadata"), and long contexts at small batch are split along the KV
axis across SMs with the partial results merged afterwards ("MLA 推理：两条计算
路径与 FlashMLA", section "decode 注意力变成了计算问题").  Which rule balances
the work is left open, so any schedule is correct that covers every page of
every request exactly once; ``check_schedule`` tests exactly that.  The library
uses one particular rule, restated in ``schedule_reference`` so that its
integer output can be compared bit for bit.  Every request is laid out on one
line of "cost" positions, F positions of segment set-up cost followed by one
position per page, and the line is cut into equal pieces, one per part:

  nb[b]   = ceil(seqlen[b] / 64)           (0 for an empty request)
  cost[b] = nb[b] + F if nb[b] > 0 else 0  (F = set-up cost of a segment, in pages)
  C[b]    = cost[0] + ... + cost[b-1]      (request b occupies positions [C[b], C[b+1]))
  page k of request b sits at position C[b] + F + k
  P_eff   = min(P, hbm_parts)              parts that already saturate HBM; with a split
            cost S > 0 (in pages), P_eff is instead whichever of min(P, hbm_parts)
            and P has the smaller estimate T + S * ceil(extra / P_eff), where
            extra counts the segments beyond one per request (ties: the smaller)
  T       = ceil(C[B] / P_eff)             positions per part
  part p takes the pages whose position lies in [p T, (p + 1) T)

Each part's pages are contiguous in (request, page) order, so a part is found
by two binary searches on C, independently of the other parts.

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


def _segments(C, nb, F, T, b):
    """Segments of request b when parts hold T positions each."""
    if nb[b] == 0:
        return 0
    return (C[b] + F + nb[b] - 1) // T - (C[b] + F) // T + 1


def schedule_reference(seqlens, num_parts: int, fixed_cost: int, hbm_parts: int, split_cost: int = 0):
    """The rule above.  Returns (meta: list of 5-tuples, num_splits: list)."""
    B = len(seqlens)
    F = fixed_cost
    nb = [pages_of(L) for L in seqlens]
    cost = [n + F if n > 0 else 0 for n in nb]
    C = [0] * (B + 1)
    for b in range(B):
        C[b + 1] = C[b] + cost[b]
    total = C[B]
    p_eff = max(1, min(num_parts, hbm_parts))
    if split_cost > 0 and total > 0 and num_parts > p_eff:
        best = None
        for pe in (p_eff, num_parts):
            T = (total + pe - 1) // pe
            extra = sum(_segments(C, nb, F, T, b) - 1 for b in range(B) if nb[b] > 0)
            est = T + split_cost * ((extra + pe - 1) // pe)
            if best is None or est < best[0]:
                best = (est, pe)
        p_eff = best[1]
    T = (total + p_eff - 1) // p_eff
    meta = []
    for p in range(num_parts):
        lo, hi = p * T, (p + 1) * T
        if total == 0 or p >= p_eff or lo >= total:
            meta.append((-1, 0, 0, 0, 0))
            continue
        # first page: request b_first is the first b with C[b + 1] > lo (never empty)
        b_first = next(b for b in range(B) if C[b + 1] > lo)
        k_first = max(0, lo - C[b_first] - F)
        if C[b_first] + F + k_first >= hi:
            meta.append((-1, 0, 0, 0, 0))      # the piece holds set-up positions only
            continue
        # last page: request b_last is the last non-empty b whose first page lies before hi
        b_last = max(b for b in range(B) if nb[b] > 0 and C[b] + F < hi)
        k_end = min(nb[b_last], hi - C[b_last] - F)
        split_first = p - (C[b_first] + F) // T
        meta.append((b_first, k_first, b_last, k_end, split_first))
    num_splits = [0] * (B + 1)
    for b in range(B):
        num_splits[b + 1] = num_splits[b] + (_segments(C, nb, F, T, b) if total > 0 else 0)
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
