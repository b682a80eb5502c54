"""The band / varlen tile schedule, checked on the host against brute force.

swa_debug_schedule returns the work items the kernels of one pass receive
(query tiles, key tiles, or the forward's pairs of query tiles), computed by
the same code the kernels run.  Brute force from the BAND
inequality (FlashAttentionVarLenScore doc, preTokens / nextTokens as the
window's left and right edges: query i sees key j iff
i - pre <= j <= i + next, local indices) gives, for every 128-row tile of
every (batch, head), the set of partner tiles holding at least one visible
pair.  The schedule must list every such tile exactly once, none outside its
sequence, with exactly that partner run, across the split of the work into
launches of at most 16 or 512 table entries; and TND entries must come
heaviest first.
"""
import numpy as np
import pytest

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry

TILE = 128

# 600 short sequences: more entries than one launch's table holds (512)
_CU600 = np.cumsum(np.random.default_rng(600).integers(1, 41, 600)).tolist()
# 40 sequences of mixed lengths, some empty and a trailing run of skipped batches
_L40 = np.random.default_rng(40).integers(0, 700, 34).tolist()
_CU40 = np.cumsum(_L40).tolist() + [0] * 6

CASES = {
    "bnsd_band": dict(layout="BNSD", B=2, N=3, D=64, S_q=1000, S_kv=1000, sparse_mode=4, pre_tokens=300,
                      next_tokens=5),
    "bnsd_long_band": dict(layout="BNSD", B=1, N=4, D=128, S_q=32768, S_kv=32768, sparse_mode=4, pre_tokens=4096,
                           next_tokens=0),
    "bnsd_nomask_rect": dict(layout="BNSD", B=1, N=2, D=64, S_q=333, S_kv=700, sparse_mode=0),
    "bnsd_rect_band": dict(layout="BNSD", B=2, N=1, D=64, S_q=300, S_kv=900, sparse_mode=4, pre_tokens=10,
                           next_tokens=500),
    "bnsd_negative_pre": dict(layout="BNSD", B=1, N=1, D=64, S_q=700, S_kv=700, sparse_mode=4, pre_tokens=-40,
                              next_tokens=300),
    "bnsd_negative_next": dict(layout="BNSD", B=1, N=2, D=64, S_q=500, S_kv=500, sparse_mode=4, pre_tokens=260,
                               next_tokens=-130),
    "bnsd_gqa": dict(layout="BNSD", B=2, N=8, N_kv=2, D=64, S_q=400, S_kv=400, sparse_mode=4, pre_tokens=150,
                     next_tokens=0),
    "tnd_600": dict(layout="TND", B=600, N=2, D=64, cu_seqlens_q=_CU600, cu_seqlens_kv=_CU600, sparse_mode=4,
                    pre_tokens=7, next_tokens=3),
    "tnd_40_mixed_skipped": dict(layout="TND", B=40, N=3, N_kv=1, D=64, cu_seqlens_q=_CU40, cu_seqlens_kv=_CU40,
                                 sparse_mode=4, pre_tokens=200, next_tokens=60),
    "tnd_rect_nomask": dict(layout="TND", B=4, N=2, D=64, cu_seqlens_q=[50, 300, 310, 310],
                            cu_seqlens_kv=[170, 180, 420, 600], sparse_mode=0),
}


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return swa.lib()


def _windows(geom, lq, lk):
    """[lo_i, hi_i] of every local query row (lo > hi: empty), by the inequality."""
    i = np.arange(lq, dtype=np.int64)
    if geom.sparse_mode == 4:
        lo = np.maximum(0, i - geom.pre_tokens)
        hi = np.minimum(lk - 1, i + geom.next_tokens)
    else:
        lo = np.zeros(lq, dtype=np.int64)
        hi = np.full(lq, lk - 1, dtype=np.int64)
    return lo, hi


def _partner_sets(geom, lq, lk):
    """{query tile: set of key tiles} and {key tile: set of query tiles} holding
    at least one visible pair."""
    lo, hi = _windows(geom, lq, lk)
    q_to_k = {t: set() for t in range((lq + TILE - 1) // TILE)}
    k_to_q = {t: set() for t in range((lk + TILE - 1) // TILE)}
    for i in range(lq):
        if lo[i] > hi[i]:
            continue
        for kt in range(lo[i] // TILE, hi[i] // TILE + 1):
            q_to_k[i // TILE].add(kt)
            k_to_q[kt].add(i // TILE)
    return q_to_k, k_to_q


def _as_run(tiles):
    if not tiles:
        return (0, 0)
    t = sorted(tiles)
    assert t == list(range(t[0], t[-1] + 1)), "partner tiles are not one run"
    return (t[0], len(t))


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("pass_", [0, 1], ids=["query_tiles", "key_tiles"])
def test_schedule_covers_every_visible_tile_once(name, pass_):
    geom = Geometry(**CASES[name])
    items = swa.swa_debug_schedule(swa.Params(geom), pass_)
    heads = geom.N if pass_ == 0 else geom.n_kv
    expect = {}
    for b, (lq, lk) in enumerate(geom.seq_lens()):
        if (lq if pass_ == 0 else lk) == 0:
            continue  # no rows on this side: no work items
        q_to_k, k_to_q = _partner_sets(geom, lq, lk)
        own = q_to_k if pass_ == 0 else k_to_q
        for h in range(heads):
            for t, partners in own.items():
                expect[(b, h, t)] = _as_run(partners)
    got = {}
    for launch, b, h, t, t0, n in items.tolist():
        key = (b, h, t)
        assert key not in got, ("listed twice", key)
        got[key] = (t0 if n else 0, n)
    assert set(got) == set(expect), (sorted(set(expect) - set(got))[:5], sorted(set(got) - set(expect))[:5])
    bad = [k_ for k_ in expect if got[k_] != expect[k_]]
    assert not bad, [(k_, got[k_], expect[k_]) for k_ in bad[:5]]
    # launches are numbered in order; each holds at most 512 table entries
    launches = items[:, 0]
    assert np.all(np.diff(launches) >= 0) and launches[0] == 0
    if geom.layout == "TND":
        n_entries = sum(1 for lq, lk in geom.seq_lens() if (lq if pass_ == 0 else lk) > 0)
        table = 16 if n_entries <= 16 else 512
        assert launches[-1] + 1 == (n_entries + table - 1) // table


@pytest.mark.parametrize("name", sorted(CASES))
def test_pair_schedule_covers_every_query_tile_once(name):
    # pass 2, the forward one CTA per pair of query tiles: pair p of each
    # (batch, head) holds query tiles 2p and 2p + 1 (the second only if it
    # exists), every tile in exactly one pair; the pair's key tiles run from
    # the first start to the last end of its tiles' brute-force partner runs
    geom = Geometry(**CASES[name])
    items = swa.swa_debug_schedule(swa.Params(geom), 2)
    expect_pairs, covered = {}, {}
    for b, (lq, lk) in enumerate(geom.seq_lens()):
        if lq == 0:
            continue
        q_to_k, _ = _partner_sets(geom, lq, lk)
        tiles = len(q_to_k)
        for h in range(geom.N):
            for t in range(tiles):
                covered[(b, h, t)] = 0
            for p in range((tiles + 1) // 2):
                runs = [_as_run(q_to_k[t]) for t in (2 * p, 2 * p + 1) if t < tiles and q_to_k[t]]
                if runs:
                    u0 = min(r[0] for r in runs)
                    expect_pairs[(b, h, p)] = (u0, max(r[0] + r[1] for r in runs) - u0)
                else:
                    expect_pairs[(b, h, p)] = (0, 0)
    got = {}
    for launch, b, h, p, t0, n in items.tolist():
        assert (b, h, p) not in got, ("pair listed twice", (b, h, p))
        got[(b, h, p)] = (t0 if n else 0, n)
        for t in (2 * p, 2 * p + 1):
            if (b, h, t) in covered:
                covered[(b, h, t)] += 1
    assert set(got) == set(expect_pairs)
    assert all(c == 1 for c in covered.values()), [k_ for k_, c in covered.items() if c != 1][:5]
    bad = [k_ for k_ in expect_pairs if got[k_] != expect_pairs[k_]]
    assert not bad, [(k_, got[k_], expect_pairs[k_]) for k_ in bad[:5]]


@pytest.mark.parametrize("name", ["tnd_600", "tnd_40_mixed_skipped", "tnd_rect_nomask"])
@pytest.mark.parametrize("pass_", [0, 1], ids=["query_tiles", "key_tiles"])
def test_tnd_entries_heaviest_first(name, pass_):
    # each sequence is one table entry; entries run in order of their
    # heaviest tile (most partner tiles), so the longest CTAs start first
    geom = Geometry(**CASES[name])
    items = swa.swa_debug_schedule(swa.Params(geom), pass_)
    order, weight = [], {}
    for _, b, _, _, _, n in items.tolist():
        if b not in weight:
            order.append(b)
            weight[b] = 0
        weight[b] = max(weight[b], n)
    w = [weight[b] for b in order]
    assert all(x >= y for x, y in zip(w, w[1:])), w[:20]


def test_schedule_rejects_bad_pass(lib):
    geom = Geometry(**CASES["bnsd_band"])
    with pytest.raises(swa.SwaError) as e:
        swa.swa_debug_schedule(swa.Params(geom), 3)
    assert e.value.status == swa.SWA_ERR_PARAM_INVALID
