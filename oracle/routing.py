"""Router top-k, combine weights and sort-free tile placement.

Oracle module (test infrastructure only). See ``oracle/__init__.py``.

Passages followed:

* "SGLang's Low-Latency Mode Boosts DeepSeek-V4.1-Flash Speed by 1.56x on
  AMD", section "NVIDIA overlaps the dependency chain", bullet "Routing
  without sorting":
  - each expert's rows go into 8-row tiles;
  - a per-expert bitmap and population counts place them, with no scan or sort;
  - the top-k choices are kept.
* "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 2.1
  (MoE router bullet). The router emits the layout that the expert
  computation consumes.

Readings where the pages are silent:

* Score function: a softmax over the k selected logits. There is no bias and
  no routed scaling factor.
* Top-k order: descending logit, and equal logits go to the lower expert id.
  The output keeps this rank order.
* Tile row order: ascending token id. This is the order a population count
  of lower bits gives. No capacity limit applies and nothing is dropped.
"""
from __future__ import annotations

import numpy as np

TILE_ROWS = 8

# ---------------------------------------------------------------- own exp (fp32)
# Cody and Waite, "Software Manual for the Elementary Functions" (1980).
# Argument reduction x = n*ln2 + r, with ln2 split into a hi part of 16
# significant bits (so n*hi is exact for |n| < 2^8) and a lo part. Then a
# Taylor polynomial of degree 8 for e^r on |r| <= ln2/2, and scaling by 2^n.
# Every step is a single correctly rounded binary32 operation (no fused
# multiply-add). A device implementation using the same operations in the
# same order returns the same bits.
_LOG2E = np.float32(1.4426950408889634)
_LN2_HI = np.float32(45426.0 / 65536.0)                         # 0.693145751953125
_LN2_LO = np.float32(0.6931471805599453 - 45426.0 / 65536.0)    # ~1.4286068e-06
_INV_FACT = [np.float32(1.0 / f) for f in (1, 1, 2, 6, 24, 120, 720, 5040, 40320)]


def exp_rn(x) -> np.ndarray:
    """e^x in binary32 for finite x <= 88, accurate to a few ulp.

    Steps, each rounded to binary32:
      n  = rint(x * log2e)                       (ties to even)
      r  = (x - n*ln2_hi) - n*ln2_lo
      p  = 1 + r*(1 + r*(1/2 + r*(1/6 + ... + r*(1/40320))))   (Horner)
      result = p * 2^n
    For n < -126 the result is p * 2^(n+64) * 2^-64: the first product is
    exact and the second rounds once into the subnormal range. For n < -150
    the result is 0.
    """
    x = np.asarray(x, dtype=np.float32)
    n = np.rint(x * _LOG2E).astype(np.float32)
    r = (x - n * _LN2_HI) - n * _LN2_LO
    p = _INV_FACT[8] * np.ones_like(r)
    for i in range(7, -1, -1):
        p = _INV_FACT[i] + r * p
    ni = n.astype(np.int32)
    out = np.empty_like(p)
    normal = ni >= -126
    out[normal] = p[normal] * np.ldexp(np.float32(1.0), ni[normal]).astype(np.float32)
    sub = (~normal) & (ni >= -150)
    if np.any(sub):
        t = p[sub] * np.ldexp(np.float32(1.0), ni[sub] + 64).astype(np.float32)
        out[sub] = t * np.float32(2.0 ** -64)
    out[ni < -150] = np.float32(0.0)
    return out


# ---------------------------------------------------------------- top-k + weights

def topk_ids(logits, k: int) -> np.ndarray:
    """The k largest logits of each row, in descending order; ties -> lower id.

    This is a plain stable sort of -logit, and the first k entries are kept.
    """
    logits = np.asarray(logits, dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def softmax_topk_weights(logits, ids) -> np.ndarray:
    """Softmax over the k selected logits of each row, in binary32.

      m   = l_1                          (the largest selected logit)
      e_j = exp_rn(l_j - m)
      s   = ((e_1 + e_2) + e_3) + ...    (rank order)
      w_j = e_j / s                      (correctly rounded divide)
    """
    logits = np.asarray(logits, dtype=np.float32)
    sel = np.take_along_axis(logits, ids.astype(np.int64), axis=1)
    d = sel - sel[:, :1]
    e = exp_rn(d)
    s = e[:, 0].copy()
    for j in range(1, e.shape[1]):
        s = s + e[:, j]
    return (e / s[:, None]).astype(np.float32)


# ---------------------------------------------------------------- placement

def placement(ids, num_experts: int):
    """Sort-free placement of (token, slot) pairs into 8-row expert tiles.

    For a token t and its j-th choice e = ids[t][j]:
      rank(t, e) = the number of tokens t' < t that also chose e
      tile = rank // 8, row = rank % 8
    This is written as a plain counting loop over tokens in ascending order.
    A population count of the bits below t in expert e's token bitmap gives
    the same rank.

    Returns a dict with:
      bitmap  uint32 [E][ceil(T/32)]  bit t of expert e set iff e in ids[t]
      counts  int32  [E]              rows placed on each expert
      tiles   int32  [E]              ceil(counts / 8)
      slot_e, slot_tile, slot_row  int32 [T][k]   where each pair went
      rows_of list of E int32 arrays  pair ids (t*k + j) in rank order
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    E = num_experts
    words = (T + 31) // 32
    bitmap = np.zeros((E, max(words, 1)), dtype=np.uint32)
    counts = np.zeros(E, dtype=np.int64)
    slot_e = np.zeros((T, k), dtype=np.int32)
    slot_tile = np.zeros((T, k), dtype=np.int32)
    slot_row = np.zeros((T, k), dtype=np.int32)
    rows_of = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            rank = int(counts[e])
            counts[e] += 1
            slot_e[t, j] = e
            slot_tile[t, j] = rank // TILE_ROWS
            slot_row[t, j] = rank % TILE_ROWS
            rows_of[e].append(t * k + j)
            bitmap[e, t // 32] |= np.uint32(1 << (t % 32))
    tiles = (counts + TILE_ROWS - 1) // TILE_ROWS
    return {
        "bitmap": bitmap,
        "counts": counts.astype(np.int32),
        "tiles": tiles.astype(np.int32),
        "slot_e": slot_e,
        "slot_tile": slot_tile,
        "slot_row": slot_row,
        "rows_of": [np.array(r, dtype=np.int32) for r in rows_of],
    }
