"""Pins for the oracle's work lists of the backward, of the candidate mask
and of the forward on CTA pairs.

``oracle/worklist.py`` enumerates the work items of the backward
(``items_bwd``, ``items_bwd_targets``), of the candidate mask
(``items_targets``, ``items_candidates``) and of CTA pairs
(``items_pairs``).  The C-ABI builders are checked
bit for bit against these lists, so the lists themselves are pinned here to
things other than themselves:

* hand-worked cases (``tests/golden/worklist_bwd_candidates_hand_cases.txt``),
  written from the rule in that file's header;
* brute force over the M-FALCON mask (HSTU paper Appendix H, Algorithm 1
  steps 4-5, ``oracle/dense.py`` ``candidate_mask``): each item's blocks
  are exactly the blocks that hold a kept pair, every kept pair is covered
  exactly once, and the order is cost descending with the stated tie-break;
* brute force over the causal mask for pair items: the two blocks' walk
  covers each causal pair exactly once;
* planted mistakes (a tie-break flip, an off-by-one in "holds a history
  key", an off-by-one in "holds a candidate row", a pair walk one block
  short) that these pins catch.
"""
import importlib.util
import os

import numpy as np
import pytest

from oracle import dense, worklist

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worklist_bwd_candidates_hand_cases.txt")
BM = 128


def _read_cases(path=GOLDEN):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case"):
            kv = dict(p.split("=") for p in line.split()[1:])
            targets = [int(x) for x in kv["targets"].split(",")] if "targets" in kv else None
            cur = {"kind": kv["kind"], "offsets": [int(x) for x in kv["offsets"].split(",")],
                   "targets": targets, "heads": int(kv["heads"]), "expect": []}
            cases.append(cur)
        else:
            cur["expect"].append([int(x) for x in line.split()])
    return cases


def _list_of(wl, case):
    """The case's list from module ``wl``: rows of (items..., hist) as lists."""
    off, heads, tg = case["offsets"], case["heads"], case["targets"]
    kind = case["kind"]
    if kind == "bwd":
        return wl.items_bwd(off, heads).tolist()
    if kind == "pairs":
        return wl.items_pairs(off, heads).tolist()
    fn = {"bwd_targets": wl.items_bwd_targets, "targets": wl.items_targets,
          "candidates": wl.items_candidates}[kind]
    it, hs = fn(off, tg, heads)
    return [list(r) + [int(h)] for r, h in zip(it.tolist(), hs.tolist())]


def test_hand_cases_cover_every_kind():
    kinds = [c["kind"] for c in _read_cases()]
    assert {"bwd", "bwd_targets", "targets", "candidates", "pairs"} <= set(kinds)
    assert len(kinds) == 14


@pytest.mark.parametrize("idx", range(14))
def test_hand_case(idx):
    case = _read_cases()[idx]
    assert _list_of(worklist, case) == case["expect"], case


# ------------------------------------------------------- brute force over the mask
def _kept(n, hist):
    """Algorithm 1's mask for one sequence (heads = 1), as a boolean (n, n)."""
    if n == 0:
        return np.zeros((0, 0), dtype=bool)
    m = dense.candidate_mask([n], [n - hist], 1, n)[0, 0]
    return m != 0.0


def _random_case(rng):
    nb = int(rng.integers(1, 6))
    lengths, targets = [], []
    for _ in range(nb):
        kind = rng.integers(0, 6)
        if kind == 0:
            n = 0
        elif kind == 1:
            n = 1
        else:
            n = int(rng.integers(1, 520))
        mode = rng.integers(0, 5)
        if n == 0 or mode == 0:
            t = 0                                  # no candidates
        elif mode == 1:
            t = n                                  # all candidates
        elif mode == 2 and n > 128:
            t = n - BM * int(rng.integers(1, (n - 1) // BM + 1))   # history a multiple of 128
        else:
            t = int(rng.integers(0, n + 1))
        lengths.append(n)
        targets.append(t)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64).tolist()
    return off, targets, int(rng.integers(1, 4))


def _fwd_walk(qt, hist):
    """The forward kernel's walk for query block qt: history blocks
    0 .. min(qt, KH) - 1, then the diagonal block."""
    kh = (hist + BM - 1) // BM
    return list(range(min(qt, kh))) + [qt]


def _bwd_walk(kt, n, hist):
    """The backward kernel's walk for key block kt: query blocks kt .. nq - 1
    when the block holds a history key, else kt alone."""
    nq = (n + BM - 1) // BM
    return list(range(kt, nq)) if BM * kt < hist else [kt]


@pytest.mark.parametrize("seed", range(40))
def test_walks_cover_each_kept_pair_once(seed):
    rng = np.random.default_rng(seed)
    off, targets, heads = _random_case(rng)
    it_f, hs_f = worklist.items_targets(off, targets, heads)
    it_b, hs_b = worklist.items_bwd_targets(off, targets, heads)
    seqs = {off[b]: (b, off[b + 1] - off[b], off[b + 1] - off[b] - targets[b])
            for b in range(len(off) - 1) if off[b + 1] > off[b]}
    for it, hs, fwd in ((it_f, hs_f, True), (it_b, hs_b, False)):
        cover = {(s0, h): np.zeros((n, n), dtype=np.int32) for s0, (_, n, _) in seqs.items()
                 for h in range(heads)}
        costs, keys = [], []
        for (s0, n, h, blk), hist in zip(it.tolist(), hs.tolist()):
            b, n_ref, hist_ref = seqs[s0]
            assert (n, hist) == (n_ref, hist_ref)
            kept = _kept(n, hist)
            walk = _fwd_walk(blk, hist) if fwd else _bwd_walk(blk, n, hist)
            for other in walk:
                qb, kb = (blk, other) if fwd else (other, blk)
                rows = slice(BM * qb, min(n, BM * qb + BM))
                cols = slice(BM * kb, min(n, BM * kb + BM))
                assert kept[rows, cols].any(), "a walked block holds no kept pair"
                cover[(s0, h)][rows, cols] += kept[rows, cols]
            # the item walks every block that holds a kept pair of its block
            nblk = (n + BM - 1) // BM
            need = [o for o in range(nblk)
                    if (kept[BM * blk:BM * blk + BM, BM * o:BM * o + BM] if fwd
                        else kept[BM * o:BM * o + BM, BM * blk:BM * blk + BM]).any()]
            assert sorted(walk) == need
            costs.append(len(need))
            keys.append((b, h, blk))
        for (s0, h), c in cover.items():
            n = c.shape[0]
            assert np.array_equal(c, _kept(n, seqs[s0][2]).astype(np.int32)), "kept pair not covered once"
        # every (sequence, head, block) once; cost descending, then b, h, block
        nblocks = sum(heads * ((n + BM - 1) // BM) for _, n, _ in seqs.values())
        assert len(set(keys)) == len(keys) == nblocks
        order = sorted(range(len(keys)), key=lambda r: (-costs[r], keys[r]))
        assert order == list(range(len(keys)))


@pytest.mark.parametrize("seed", range(40))
def test_causal_backward_walks_cover_each_pair_once(seed):
    rng = np.random.default_rng(100 + seed)
    off, _, heads = _random_case(rng)
    it = worklist.items_bwd(off, heads)
    zero = [0] * (len(off) - 1)
    it_t, hs_t = worklist.items_bwd_targets(off, zero, heads)
    # without candidates the candidate backward's list is the causal one
    assert np.array_equal(it, it_t)
    for (s0, n, h, kt) in it.tolist():
        tri = np.tril(np.ones((n, n), dtype=bool))
        need = [qb for qb in range((n + BM - 1) // BM) if tri[BM * qb:BM * qb + BM, BM * kt:BM * kt + BM].any()]
        assert need == list(range(kt, (n + BM - 1) // BM))


@pytest.mark.parametrize("seed", range(40))
def test_candidates_only_are_the_blocks_with_candidate_rows(seed):
    rng = np.random.default_rng(200 + seed)
    off, targets, heads = _random_case(rng)
    it, hs = worklist.items_targets(off, targets, heads)
    ic, hc = worklist.items_candidates(off, targets, heads)
    want = []
    for r, ((s0, n, h, qt), hist) in enumerate(zip(it.tolist(), hs.tolist())):
        rows = np.arange(BM * qt, min(n, BM * qt + BM))
        if np.any(rows >= hist):
            want.append(r)
    assert np.array_equal(ic, it[want].reshape(-1, 4))
    assert np.array_equal(hc, hs[want])


# ----------------------------------------------------------- planted mistakes
MUTANTS = {
    # ties broken by head before sequence in the causal backward
    "bwd_tie_break": ("rows.append((-(nq - kt), b, h, kt, offsets[b], n))",
                      "rows.append((-(nq - kt), h, b, kt, offsets[b], n))"),
    # ties broken by key block descending in the candidate backward
    "bwd_targets_tie_break": ("rows.append((-cost, b, h, kt, offsets[b], n, hist))",
                              "rows.append((-cost, b, h, -kt, offsets[b], n, hist))"),
    # key hist counted as a history key
    "history_key_off_by_one": ("any(j < hist for j in", "any(j <= hist for j in"),
    # row hist not counted as a candidate row
    "candidate_row_off_by_one": ("any(hs[r] <= i < it[r, 1]", "any(hs[r] < i < it[r, 1]"),
    # a pair's walk counted one block short
    "pair_cost_off_by_one": ("rows.append((-min(2 * qp + 2, nq), b, h, qp, offsets[b], n))",
                             "rows.append((-min(2 * qp + 1, nq), b, h, qp, offsets[b], n))"),
}


def _mutant_module(tmp_path, name):
    src = open(worklist.__file__).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"worklist_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"worklist_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _hand_cases_pass(wl) -> bool:
    return all(_list_of(wl, c) == c["expect"] for c in _read_cases())


def test_committed_worklist_passes_the_hand_cases():
    assert _hand_cases_pass(worklist)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert not _hand_cases_pass(_mutant_module(tmp_path, name)), name


@pytest.mark.parametrize("seed", range(30))
def test_pair_walks_cover_each_causal_pair_once(seed):
    # Every kept (causal) pair of a sequence lies in exactly one walked
    # (query block, key block) of exactly one pair item, every walked key
    # block holds a kept pair of one of the pair's two blocks, and the cost
    # is the number of key blocks walked.
    rng = np.random.default_rng(300 + seed)
    off, _, heads = _random_case(rng)
    it = worklist.items_pairs(off, heads)
    seqs = {off[b]: (b, off[b + 1] - off[b]) for b in range(len(off) - 1) if off[b + 1] > off[b]}
    cover = {(s0, h): np.zeros((n, n), dtype=np.int32) for s0, (_, n) in seqs.items() for h in range(heads)}
    costs, keys = [], []
    for s0, n, h, qp in it.tolist():
        b, n_ref = seqs[s0]
        assert n == n_ref
        tri = np.tril(np.ones((n, n), dtype=bool))
        nq = (n + BM - 1) // BM
        walk = list(range(min(2 * qp + 1, nq - 1) + 1))
        rows = slice(2 * BM * qp, min(n, 2 * BM * qp + 2 * BM))
        assert rows.start < n
        for kb in walk:
            cols = slice(BM * kb, min(n, BM * kb + BM))
            assert tri[rows, cols].any(), "a walked key block holds no kept pair"
            cover[(s0, h)][rows, cols] += tri[rows, cols]
        need = [kb for kb in range(nq) if tri[rows, BM * kb:BM * kb + BM].any()]
        assert walk == need
        costs.append(len(walk))
        keys.append((b, h, qp))
    for (s0, h), c in cover.items():
        n = c.shape[0]
        assert np.array_equal(c, np.tril(np.ones((n, n), dtype=np.int32)))
    assert len(set(keys)) == len(keys)
    order = sorted(range(len(keys)), key=lambda r: (-costs[r], keys[r]))
    assert order == list(range(len(keys)))
