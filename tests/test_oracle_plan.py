"""The chunk plan and bucket assignment against torch.chunk itself (the library call the
page's dynamic_chunk makes) and against invariants of the table."""
import numpy as np
import torch


def _page_dynamic_chunk(t):
    """The page's dynamic_chunk on a CPU tensor, evaluated with the real torch.chunk."""
    nbytes = t.numel() * t.element_size()
    return torch.chunk(t, max(1, nbytes // (128 * 1024 - (128 * 1024) % 64)))


def test_plan_matches_torch_chunk_dense_range(orc):
    # every n in [0, 300000) for fp32 and fp16, plus a log-spaced sample up to 2^28
    for eb, dtype in ((4, torch.float32), (2, torch.float16)):
        base = torch.empty(300000, dtype=dtype)
        for n in range(0, 300000, 7 if eb == 4 else 11):
            pieces = _page_dynamic_chunk(base[:n])
            k, c = orc.bucket_chunks(n, eb)
            assert k == len(pieces), (n, eb)
            assert c == pieces[0].numel(), (n, eb)


def test_plan_matches_torch_chunk_large(orc):
    rng = np.random.default_rng(5)
    sizes = sorted(set(int(x) for x in np.exp(rng.uniform(np.log(1), np.log(2 ** 28), 400))))
    sizes += [2 ** k + d for k in (12, 16, 20, 24, 28) for d in (-1, 0, 3, 17)] + [1000003]
    big = torch.empty(2 ** 28 + 17, dtype=torch.float32)
    for n in sizes:
        pieces = _page_dynamic_chunk(big[:n])
        off = orc.plan_chunks([n], 4)
        assert len(off) - 1 == len(pieces)
        assert list(np.diff(off)) == [p.numel() for p in pieces], n


def test_plan_fewer_pieces_than_requested(orc):
    """A 5.24 GB fp32 bucket asks for k = 40000 pieces; torch.chunk returns 39999.  The
    tensor is never touched, so its pages are never backed."""
    n = 40000 * 32768 + 1
    t = torch.empty(n, dtype=torch.float32)
    pieces = _page_dynamic_chunk(t)
    assert orc.bucket_chunks(n, 4) == (len(pieces), pieces[0].numel()) == (39999, 32769)
    off = orc.plan_chunks([n], 4)
    assert list(np.diff(off[-3:])) == [p.numel() for p in pieces[-2:]]


def test_plan_multi_bucket_table(orc):
    rng = np.random.default_rng(9)
    for eb in (2, 4):
        buckets = [int(x) for x in rng.integers(0, 200000, 12)] + [0, 65536, 1]
        off = orc.plan_chunks(buckets, eb)
        assert off[0] == 0 and off[-1] == sum(buckets)
        assert np.all(np.diff(off) >= 0)
        # each bucket's slice of the table is that bucket's own dynamic_chunk, rebased
        pos, start = 0, 0
        for n in buckets:
            k, _ = orc.bucket_chunks(n, eb)
            sub = off[pos:pos + k + 1] - start
            assert list(sub) == list(orc.plan_chunks([n], eb)), n
            pos += k
            start += n
        assert pos == len(off) - 1


def test_payload_reduction_75_percent(orc):
    """int8 codes plus one fp32 scale per chunk against fp32 values: 1 - (n + 4k) / 4n
    lies in [0.7499, 0.75] for every bucket of at least 128 KiB (about 75% fewer bytes)."""
    for n in [32768, 262144, 6553600, 60192808, 2 ** 28, 1000003, 2 ** 20 + 17]:
        k, _ = orc.bucket_chunks(n, 4)
        saving = 1 - (n + 4 * k) / (4 * n)
        assert 0.7499 <= saving <= 0.75, (n, saving)


def test_bucket_greedy_is_maximal(orc):
    """Every bucket is within the cap unless it holds one tensor, and no bucket could have
    taken the first tensor of the next one."""
    rng = np.random.default_rng(3)
    cap = 25 * 1024 * 1024
    for eb in (2, 4):
        sizes = [int(x) for x in np.round(np.exp(rng.uniform(np.log(64), np.log(2359296), 300)))]
        bot, be = orc.assign_buckets(sizes, eb, cap)
        assert sum(be) == sum(sizes)
        for b in range(len(be)):
            members = [s for s, k in zip(sizes, bot) if k == b]
            assert be[b] * eb <= cap or len(members) == 1
            if b + 1 < len(be):
                nxt = next(s for s, k in zip(sizes, bot) if k == b + 1)
                assert (be[b] + nxt) * eb > cap


def _page_dynamic_chunk_sized(t, chunk_size):
    """The page's dynamic_chunk with its CHUNK_SIZE knob set to chunk_size, on the real
    torch.chunk (alignment 64 as on the page)."""
    nbytes = t.numel() * t.element_size()
    return torch.chunk(t, max(1, nbytes // (chunk_size - chunk_size % 64)))


def test_plan_sized_matches_torch_chunk(orc):
    """Other base chunk sizes, including ones that are not multiples of the 64-byte alignment
    (so the page's `chunk_size - chunk_size % alignment` term matters)."""
    rng = np.random.default_rng(21)
    base = torch.empty(2 ** 22, dtype=torch.float32)
    for chunk_size in (100, 4096, 16384, 32868, 65536, 131072, 262144, 1048576, 1000003):
        sizes = sorted(set(int(x) for x in np.exp(rng.uniform(0, np.log(2 ** 22), 150)))) + [0, 1, 2 ** 22]
        for eb, dtype in ((4, torch.float32), (2, torch.float16)):
            t = base.view(dtype) if eb == 4 else base.view(torch.float16)
            for n in sizes:
                pieces = _page_dynamic_chunk_sized(t[:n], chunk_size)
                k, c = orc.bucket_chunks_sized(n, eb, chunk_size)
                assert k == len(pieces), (chunk_size, n, eb)
                assert c == pieces[0].numel(), (chunk_size, n, eb)
        off = orc.plan_chunks_ex(sizes, 4, orc.SCOPE_CHUNK, chunk_size)
        pos = 0
        for n in sizes:
            k, c = orc.bucket_chunks_sized(n, 4, chunk_size)
            assert off[pos + 1] - off[pos] == c or (n == 0 and c == 0)
            pos += k
        assert pos == len(off) - 1 and off[-1] == sum(sizes)


def test_plan_default_chunk_size_is_the_page_plan(orc):
    rng = np.random.default_rng(23)
    buckets = [int(x) for x in rng.integers(0, 9_000_000, 20)] + [0, 1, 32768]
    for eb in (2, 4):
        assert np.array_equal(orc.plan_chunks_ex(buckets, eb, orc.SCOPE_CHUNK, 128 * 1024),
                              orc.plan_chunks(buckets, eb))


def test_plan_whole_bucket_and_whole_tensor_scopes(orc):
    """One scale per bucket or per tensor: the table is the entries' boundaries, one chunk per
    entry, an empty entry an empty chunk."""
    sizes = [64, 0, 2359296, 1, 0, 513, 6553600, 3]
    want = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    for scope in (orc.SCOPE_BUCKET, orc.SCOPE_TENSOR):
        for eb in (2, 4):
            assert np.array_equal(orc.plan_chunks_ex(sizes, eb, scope), want)


def test_plan_ex_rejects_bad_arguments(orc):
    import pytest
    with pytest.raises(ValueError):
        orc.plan_chunks_ex([10], 4, 3)
    with pytest.raises(ValueError):
        orc.plan_chunks_ex([10], 4, orc.SCOPE_CHUNK, 63)   # aligned part 0
    with pytest.raises(ValueError):
        orc.plan_chunks_ex([-1], 4, orc.SCOPE_TENSOR)
