"""Index arithmetic of the routing kernel's score tiles, checked on the host.

The routing kernel stages 128 video key means at a time and scores them with
a tile of QPT query blocks x KPT keys per thread (256 threads; thread tid is
query group tid // NKG and key group tid % NKG, NKG = 256 / (QB / QPT)); a
short last chunk takes a tile with one key per thread.  These tests restate
that mapping and the chunk-length rule that picks the tile, for every
launcher variant, and check for every chunk length that each (query block,
key) pair of the chunk is scored by exactly one thread and that no thread
reads a staged row past the 128 rows of the chunk buffer.
"""
import pytest

THREADS = 256
CHUNK = 128
# (QB, QPT, KPT) of the launcher's variants
VARIANTS = [(32, 8, 2), (16, 4, 2), (8, 4, 1), (4, 2, 1)]


def tile_for(qb, qpt, kpt, nk):
    """The tile the kernel uses for a chunk of nk keys (nk <= 128)."""
    if nk == CHUNK:
        return qpt, kpt
    if qb % 2 == 0 and nk <= THREADS * 2 // qb and qpt > 2:
        return 2, 1
    if qb % 4 == 0 and nk <= THREADS * 4 // qb and qpt > 4:
        return 4, 1
    if qb % 8 == 0 and nk <= THREADS * 8 // qb and (qpt > 8 or kpt > 1):
        return 8, 1
    return qpt, kpt


def scored_pairs(qb, qpt, kpt, nk):
    """(query, key) pairs each thread writes, and the staged rows it reads."""
    nqg = qb // qpt
    nkg = THREADS // nqg
    writes, rows = [], []
    for tid in range(THREADS):
        kg, qg = tid % nkg, tid // nkg
        if kg >= nk:  # no key of this chunk: the thread returns
            continue
        for e in range(kpt):
            rows.append(kg + nkg * e)
            j = kg + nkg * e
            if j < nk:
                writes += [(qg * qpt + q, j) for q in range(qpt)]
    return writes, rows


@pytest.mark.parametrize("qb,qpt,kpt", VARIANTS)
def test_full_tile_shape(qb, qpt, kpt):
    # the full-chunk tile covers exactly the 128 staged keys
    assert (THREADS // (qb // qpt)) * kpt == CHUNK


@pytest.mark.parametrize("qb,qpt,kpt", VARIANTS)
def test_every_pair_once_in_bounds(qb, qpt, kpt):
    for nk in range(1, CHUNK + 1):
        tq, tk = tile_for(qb, qpt, kpt, nk)
        assert qb % tq == 0
        writes, rows = scored_pairs(qb, tq, tk, nk)
        assert len(writes) == len(set(writes)), (nk, tq, tk)
        assert set(writes) == {(q, j) for q in range(qb) for j in range(nk)}, (nk, tq, tk)
        assert max(rows) < CHUNK, (nk, tq, tk)


def test_short_chunk_keeps_threads_busy():
    # H3: 144 video blocks, a last chunk of 16 keys; every thread scores
    # two pairs instead of 32 threads scoring sixteen each
    tq, tk = tile_for(32, 8, 2, 16)
    assert (tq, tk) == (2, 1)
    nkg = THREADS // (32 // tq)
    busy = sum(1 for tid in range(THREADS) if tid % nkg < 16)
    assert busy == THREADS
