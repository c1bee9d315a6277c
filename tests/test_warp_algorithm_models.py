"""CPU models of two warp-level algorithms the kernels rely on (host logic;
no GPU), checked against their definitions.

* The reduce-scatter of the decode attention kernel: 32 lanes each hold N
  values (N a power of two); at offsets 16, 8, ... a lane keeps one half of
  its remaining values and adds the partner lane's other half, then plain
  butterflies once one value is left.  Lane l must end with the warp total
  of value l / (32 / N).
* The one-token expert selection (routers of up to 256 experts): lane l
  holds the order keys of experts l, l + 32, ...; each of the K rounds takes
  the lane's best key by a tree of adjacent pairs (left wins ties), the
  warp's largest key (redux max) and the lowest expert holding it (redux
  min), then clears that key.  The result must be the oracle's top-K
  (larger logit first, equal logits to the lower expert), including
  bitwise ties inside one lane and across lanes, -0 equal to +0.
"""
import numpy as np
import pytest

import oracle


# ---------------------------------------------------------------- reduce-scatter
def _reduce_scatter(vals):
    """vals[lane][j], 32 lanes x N values -> the value each lane returns."""
    v = [list(map(float, row)) for row in vals]
    N = len(v[0])
    n = N
    o = 16
    while o > 0:
        nxt = [row[:] for row in v]
        for lane in range(32):
            partner = lane ^ o
            if n > 1:
                up = (lane & o) != 0
                half = n // 2
                for j in range(half):
                    # the partner sends what it does not keep: its v[j] if it is "up", else v[j + half]
                    p_up = (partner & o) != 0
                    send_from_partner = v[partner][j] if p_up else v[partner][j + half]
                    keep = v[lane][j + half] if up else v[lane][j]
                    nxt[lane][j] = keep + send_from_partner
            else:
                nxt[lane][0] = v[lane][0] + v[partner][0]
        v = nxt
        if n > 1:
            n //= 2
        o >>= 1
    return [row[0] for row in v]


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 32])
def test_reduce_scatter_lane_mapping(N):
    rng = np.random.default_rng(N)
    # small integers: every sum is exact, so equality is the check
    vals = rng.integers(-1000, 1000, size=(32, N)).astype(np.float64)
    got = _reduce_scatter(vals)
    totals = vals.sum(axis=0)
    for lane in range(32):
        assert got[lane] == totals[lane // (32 // N)], (N, lane)


# ---------------------------------------------------------------- one-token selection
def _order_key(f):
    """Float32 -> uint32 with the order of the values (-0 and +0 equal); 0 is
    reserved for absent or taken (present keys are at least 1)."""
    b = int(np.array([np.float32(f) + np.float32(0.0)], np.float32).view(np.uint32)[0])
    k = (~b & 0xFFFFFFFF) if b & 0x80000000 else (b | 0x80000000)
    return max(k, 1)


def _select_single(logits, K):
    E = len(logits)
    per = max(2, 1 << int(np.ceil(np.log2(max(1, (E + 31) // 32)))))
    key = [[_order_key(logits[j * 32 + lane]) if j * 32 + lane < E else 0 for j in range(per)] for lane in range(32)]
    out = []
    for _ in range(K):
        lane_best = []
        for lane in range(32):
            tk, tj = key[lane][:], list(range(per))
            w = 1
            while w < per:
                for j in range(0, per - w, 2 * w):
                    if tk[j + w] > tk[j]:
                        tk[j], tj[j] = tk[j + w], tj[j + w]
                w *= 2
            lane_best.append((tk[0], tj[0]))
        kmax = max(b for b, _ in lane_best)
        emin = min((j * 32 + lane) if (b == kmax and kmax != 0) else 0xFFFFFFFF
                   for lane, (b, j) in enumerate(lane_best))
        key[emin & 31][emin >> 5] = 0
        out.append(emin)
    return out


@pytest.mark.parametrize("E,K", [(1, 1), (7, 3), (33, 8), (64, 4), (200, 8), (256, 8), (256, 16)])
def test_one_token_selection_matches_oracle_rule(E, K):
    rng = np.random.default_rng(E * 31 + K)
    for trial in range(20):
        logits = rng.standard_normal(E).astype(np.float32)
        if trial % 4 == 1:  # bitwise ties across lanes and inside one lane
            for e in rng.choice(E, size=min(E, 6), replace=False):
                logits[e] = logits[0]
        if trial % 4 == 2:  # -0 and +0 tie
            logits[rng.integers(E)] = np.float32(-0.0)
            logits[rng.integers(E)] = np.float32(0.0)
        if trial % 4 == 3:  # all equal: experts 0..K-1
            logits[:] = np.float32(0.5)
        ref = oracle.topk_select(logits.astype(np.float64)[None, :], min(K, E))[0].tolist()
        assert _select_single(logits, min(K, E)) == ref, (E, K, trial)
