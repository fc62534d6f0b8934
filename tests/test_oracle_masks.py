"""Pins of the oracle's mask predicate (CPU only).

* literal hand-written matrices from the pages' stated rules (tests/golden);
* the vectorised builder against brute-force enumeration of the predicate;
* special cases: W >= S gives the plain lower triangle, no pad and no image
  gives a band of width W.
"""

import os

import numpy as np
import pytest

from oracle import masks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "masks_s6_w3.txt")


def _load_golden():
    cases, name, meta, rows = [], None, None, []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            if name:
                cases.append((name, meta, np.array(rows, dtype=bool)))
            name, meta, rows = line[1:-1], None, []
        elif meta is None:
            meta = dict(kv.split("=") for kv in line.split())
        else:
            rows.append([c == "1" for c in line])
    cases.append((name, meta, np.array(rows, dtype=bool)))
    return cases


CASES = _load_golden()


@pytest.mark.parametrize("name,meta,expected", CASES, ids=[c[0] for c in CASES])
def test_literal_masks(name, meta, expected):
    n = expected.shape[0]
    w = int(meta["window"])
    vs = int(meta["valid_start"])
    img = [int(x) for x in meta["img"].split(",")]
    doc = [int(x) for x in meta["doc"].split(",")]
    got = masks.prefill_mask(n, w, vs, img, doc)
    assert np.array_equal(got, expected), f"{name}\n{got.astype(int)}"
    assert np.array_equal(masks.prefill_mask_loops(n, w, vs, img, doc), expected)


def test_golden_file_has_all_cases():
    assert {c[0] for c in CASES} >= {"causal_window", "doc_causal_two_docs",
                                     "vlm_block_of_3_future_pair",
                                     "vlm_block_of_5_old_pair_rejected", "left_padding_two"}


@pytest.mark.parametrize("seed", range(8))
def test_vectorised_equals_bruteforce(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(5, 24))
    w = int(rng.integers(1, n + 2))
    vs = int(rng.integers(0, 4))
    img = np.full(n, -1)
    nid = 0
    pos = int(rng.integers(0, 3))
    while pos < n - 1:
        if rng.random() < 0.5:
            ln = int(rng.integers(1, 7))
            img[pos:pos + ln] = nid
            nid += 1
            pos += ln
        pos += int(rng.integers(1, 4))
    cuts = sorted(rng.choice(np.arange(1, n), size=int(rng.integers(0, 3)), replace=False).tolist())
    doc = np.zeros(n, dtype=np.int64)
    for c in cuts:
        doc[c:] += 1
    got = masks.prefill_mask(n, w, vs, img, doc)
    exp = masks.prefill_mask_loops(n, w, vs, img, doc)
    assert np.array_equal(got, exp)
    rows = rng.choice(n, size=4, replace=False)
    assert np.array_equal(masks.prefill_mask(n, w, vs, img, doc, rows=rows), exp[rows])


def test_wide_window_is_lower_triangle():
    for n in (1, 7, 33):
        assert np.array_equal(masks.prefill_mask(n, n + 5), np.tril(np.ones((n, n), dtype=bool)))


def test_band_without_pad_or_images():
    n, w = 40, 9
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    band = (j <= i) & (i - j < w)
    assert np.array_equal(masks.prefill_mask(n, w), band)
    assert masks.prefill_mask(n, w).sum(axis=1).max() == w


def test_doc_ids_from_cu_seqlens():
    doc = masks.doc_ids_from_cu_seqlens([0, 3, 3, 7], 7)
    assert doc.tolist() == [0, 0, 0, 2, 2, 2, 2]
    with pytest.raises(ValueError):
        masks.doc_ids_from_cu_seqlens([0, 3], 5)


def test_decode_mask_full_matches_predicate():
    for p in range(10, 30):
        for vs in (0, 3, 12):
            pos = np.arange(-3, p + 3)
            got = masks.decode_mask_full(p, 7, vs, pos)
            exp = np.array([k >= 0 and masks.allowed(p, k, 7, vs) for k in pos])
            assert np.array_equal(got, exp)
