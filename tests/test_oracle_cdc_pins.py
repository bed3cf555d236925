"""Pins of the oracle's content-defined chunking (Irminsul §2.2, content hash
keying with CDC): Gear rolling hash over 64-token windows, chunk ends where
the hash falls below a threshold, xxHash64 fingerprints.

Each pin checks the oracle against something other than itself: published
values of the two named algorithms, an independent installed implementation
of XXH64, the windowed closed form of the Gear recurrence, and the property
the pages ask of content-defined boundaries (they follow the content, not
its offset)."""
import ctypes as C
import ctypes.util

import numpy as np
import pytest

import synth

M64 = 2**64 - 1


def _libxxhash():
    for name in ("libxxhash.so.0", ctypes.util.find_library("xxhash")):
        if not name:
            continue
        try:
            lib = C.CDLL(name)
        except OSError:
            continue
        lib.XXH64.restype = C.c_uint64
        lib.XXH64.argtypes = [C.c_void_p, C.c_size_t, C.c_uint64]
        return lib
    return None


def test_xxh64_published_empty_input_value(oracle):
    # the value the xxHash specification's reference implementation gives
    # for zero bytes with seed 0
    assert oracle.xxh64(b"", 0) == 0xEF46DB3751D8E999


def test_splitmix64_published_first_outputs(oracle):
    # the first outputs of SplitMix64 seeded with 0, as printed by the
    # public-domain reference code (Vigna, splitmix64.c)
    assert oracle.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert oracle.splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert oracle.splitmix64_at(0, 2) == 0x06C45D188009454F


def test_xxh64_matches_the_installed_library(oracle):
    lib = _libxxhash()
    if lib is None:
        pytest.skip("libxxhash not installed")
    rng = np.random.default_rng(7)
    # every code path: < 32 bytes, whole stripes, 8/4/1-byte tails, long input
    for n in list(range(0, 72)) + [96, 127, 128, 129, 1000, 4099]:
        for seed in (0, 1, 0x9E3779B97F4A7C15, M64):
            d = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
            buf = C.create_string_buffer(d, max(1, n))
            assert oracle.xxh64(d, seed) == lib.XXH64(C.cast(buf, C.c_void_p), n, seed), (n, seed)


def test_gear_hash_is_the_64_token_window_sum(oracle):
    # h(i) = sum over the last 64 tokens of G(x_{i-k}) * 2^k mod 2^64, with G
    # the SplitMix64 output numbered by the token id (big-integer arithmetic)
    rng = np.random.default_rng(3)
    toks = rng.integers(0, 129280, 300).astype(np.int32)
    seed = 12345
    g = [oracle.splitmix64_at(seed, int(t)) for t in toks]
    h = oracle.gear_hashes(toks, seed)
    for i in range(len(toks)):
        want = sum(g[i - k] << k for k in range(min(i + 1, 64))) & M64
        assert int(h[i]) == want, i


def _chunks(oracle, ts, gear_seed, threshold, fp_seed=0):
    ends, fps, n = oracle.cdc(ts.stream_off, ts.tokens, gear_seed, threshold, fp_seed)
    assert n == len(ends)
    return ends, fps


def test_chunks_tile_each_stream_and_fingerprints_name_their_tokens(oracle):
    ts = synth.token_streams(11, [0, 1, 63, 64, 65, 700, 0, 5000], shared_segments=2,
                             segment_lo=40, segment_hi=200)
    ends, fps = _chunks(oracle, ts, 99, 1 << 58)
    # ends are increasing, every non-empty stream's end is a chunk end, and no
    # chunk crosses a stream end
    assert np.all(np.diff(ends) > 0)
    off = ts.stream_off
    stream_ends = {int(off[s + 1]) for s in range(ts.num_streams) if off[s + 1] > off[s]}
    assert stream_ends <= set(int(e) for e in ends)
    starts = np.concatenate([[0], ends[:-1]])
    for a, b in zip(starts, ends):
        s = int(np.searchsorted(off, a, side="right") - 1)
        assert off[s] <= a < b <= off[s + 1]
    # every stream is chunked on its own: its ends are where the windowed
    # hash of that stream alone (pinned to the closed form above) falls below
    # the threshold, plus its end
    for q in range(ts.num_streams):
        a, b = int(off[q]), int(off[q + 1])
        h = oracle.gear_hashes(ts.tokens[a:b], 99)
        want = sorted({a + i + 1 for i in np.nonzero(h < np.uint64(1 << 58))[0]} |
                      ({b} if b > a else set()))
        assert [int(e) for e in ends if a < e <= b] == want, q
    # each fingerprint is XXH64 of the chunk's ids as little-endian words
    for a, b, f in zip(starts, ends, fps):
        assert int(f) == oracle.xxh64(ts.tokens[a:b].astype("<u4").tobytes(), 0)
    assert np.array_equal(oracle.fingerprint(starts, ends, ts.tokens, 0), fps)


def test_chunk_ends_follow_content_not_offset(oracle):
    # Irminsul §2.2: boundaries align with the content.  Prepending any prefix
    # of at least 64 tokens leaves every boundary that lies 64 or more tokens
    # into the original stream where it was (shifted by the prefix), with the
    # same fingerprints for the chunks that do not cross the junction.
    base = synth.token_streams(5, [20000]).tokens
    thr = 1 << 57
    a_ends, a_fps = _chunks(oracle, synth.TokenStreams(np.array([0, len(base)]), base), 7, thr)
    for plen in (64, 97, 1000):
        pre = synth.token_streams(100 + plen, [plen]).tokens
        both = np.concatenate([pre, base])
        b_ends, b_fps = _chunks(oracle, synth.TokenStreams(np.array([0, len(both)]), both), 7, thr)
        a_set = {int(e) + plen: f for e, f in zip(a_ends, a_fps) if e >= 64}
        b_set = {int(e): f for e, f in zip(b_ends, b_fps) if e >= plen + 64}
        assert set(a_set) == set(b_set)
        keys = sorted(a_set)
        for k0, k1 in zip(keys, keys[1:]):  # whole chunks past the first boundary
            assert a_set[k1] == b_set[k1]


def test_threshold_sets_the_mean_chunk_length(oracle):
    ts = synth.token_streams(8, [1 << 20])
    for log_len in (6, 8, 10):
        ends, _ = _chunks(oracle, ts, 1, 1 << (64 - log_len))
        mean = (1 << 20) / len(ends)
        assert 0.9 * (1 << log_len) < mean < 1.1 * (1 << log_len), (log_len, mean)


def test_threshold_extremes_and_capacity(oracle):
    ts = synth.token_streams(9, [50, 0, 70])
    ends, _ = _chunks(oracle, ts, 1, 0)             # nothing falls below 0
    assert ends.tolist() == [50, 120]
    ends, _ = _chunks(oracle, ts, 1, M64)           # everything but h = 2^64 - 1
    assert ends.tolist() == list(range(1, 121))
    e, f, n = oracle.cdc(ts.stream_off, ts.tokens, 1, M64, 0, max_chunks=10)
    assert n == 120 and e.tolist() == list(range(1, 11))


def test_seeds_change_boundaries_and_fingerprints(oracle):
    ts = synth.token_streams(12, [4000])
    e1, f1 = _chunks(oracle, ts, 1, 1 << 58, 0)
    e2, _ = _chunks(oracle, ts, 2, 1 << 58, 0)
    _, f3 = _chunks(oracle, ts, 1, 1 << 58, 5)
    assert e1.tolist() != e2.tolist()
    assert not np.any(f1 == f3)
