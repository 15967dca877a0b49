"""The reading the truncated verify's and DRIFT's selections rest on, checked
on the host (no GPU): with a row cut into chunks, the k-th largest chunk
maximum is at most the row's k-th largest logit, so every logit that top-k
keeps lies in a chunk whose maximum reaches it; and the k-th largest of any
grouping's group maxima (the selection kernel's lower bound over its
threads' largest maxima) is at most that.  The chunks are laid out as the
ring stream's consumer threads hold them: tile t of 1024 16-byte vectors,
thread i holding vectors i, i + 256, i + 512 and i + 768.  Keys are the top 16
bits of the order key, as the stream stores them."""
import numpy as np
import pytest

from workloads import synthetic as S


def order_key32(x):
    """Order-preserving 32-bit key of float32 values (larger value, larger key)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    neg = (u & 0x80000000) != 0
    return np.where(neg, (~u) & 0xFFFFFFFF, u | 0x80000000).astype(np.uint64)


def chunk_of(V, epv):
    """Chunk id of every element of a row (tile t, consumer thread i)."""
    per_tile = 256 * 4 * epv
    idx = np.arange(V)
    t, within = idx // per_tile, idx % per_tile
    vec = within // epv
    return t * 256 + vec % 256


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("k", [1, 32, 50, 64, 256])
def test_kth_chunk_maximum_bounds_the_kth_logit(dtype, k):
    rng = np.random.default_rng(k)
    for trial in range(6):
        V = int(rng.choice([4099, 20000, 128256]))
        x = rng.normal(0, 3, V).astype(np.float32)
        if trial % 3 == 1:  # ties straddling the boundary
            x = np.minimum(x, 6.0)
            x[rng.choice(V, 200, replace=False)] = 6.0
        if trial % 3 == 2:  # a coarse row: many equal values
            x = np.round(x)
        if dtype == "bf16":
            x = S.bf16_bits_to_f32(S.f32_to_bf16_bits(x))
        epv = 8 if dtype == "bf16" else 4
        key = order_key32(x)
        key16 = key >> 16
        ch = chunk_of(V, epv)
        nch = ch.max() + 1
        cmax = np.zeros(nch, np.uint64)
        np.maximum.at(cmax, ch, key16)
        th = np.sort(cmax)[::-1][k - 1]
        kth = np.sort(key)[::-1][k - 1]
        assert th <= (kth >> 16)
        kept = key >= kth  # top-k with boundary ties
        assert np.all(cmax[ch[kept]] >= th)
        # the candidates: every logit whose key reaches th, all in chunks reaching th
        cand = key16 >= th
        assert np.all(cmax[ch[cand]] >= th)
        assert np.all(cand[kept])
        # a lower bound over any grouping of the maxima (192 groups, strided)
        for groups in (192, 37):
            gmax = np.zeros(groups, np.uint64)
            np.maximum.at(gmax, np.arange(nch) % groups, cmax)
            if k <= groups:
                lb = np.sort(gmax)[::-1][k - 1]
                assert lb <= th


def test_flat_row_sends_every_chunk_past_the_limit():
    """An all-equal row ties every chunk maximum: more chunks than the
    selection re-reads (256) reach the threshold, which sends the row to the
    whole-row search."""
    V = 128256
    x = np.full(V, 1.25, np.float32)
    key16 = order_key32(x) >> 16
    ch = chunk_of(V, 8)
    cmax = np.zeros(ch.max() + 1, np.uint64)
    np.maximum.at(cmax, ch, key16)
    th = np.sort(cmax)[::-1][49]
    assert (cmax >= th).sum() > 256
