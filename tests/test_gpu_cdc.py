"""Content-defined chunking on the GPU (kv_cdc, kv_fingerprint) against the
oracle: chunk ends, chunk counts and fingerprints are integers, compared bit
for bit (Irminsul §2.2, content hash keying with CDC and the fixed-window
fallback)."""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth

pytestmark = pytest.mark.gpu

M64 = 2**64 - 1


@pytest.fixture(scope="module")
def orc():
    kv.load()
    return O.get()


def _run(ts, gear_seed, threshold, fp_seed=0, max_chunks=None):
    total = len(ts.tokens)
    cap = total if max_chunks is None else max_chunks
    off = torch.from_numpy(ts.stream_off).cuda()
    tok = torch.from_numpy(ts.tokens).cuda()
    ends = torch.full((max(cap, 1),), -1, dtype=torch.int64, device="cuda")
    fps = torch.zeros((max(cap, 1),), dtype=torch.int64, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(kv.kv_cdc_workspace_size(total), 256), dtype=torch.uint8, device="cuda")
    kv.kv_cdc(ts.num_streams, off, total, tok, gear_seed, threshold, fp_seed, cap, ends, fps,
              cnt, ws)
    status = kv.kv_get_device_status(ws)
    n = int(cnt.item())
    k = min(n, cap)
    return (status, n, ends[:k].cpu().numpy(),
            fps[:k].cpu().numpy().view(np.uint64))


def _check(orc, ts, gear_seed, threshold, fp_seed=0):
    status, n, ends, fps = _run(ts, gear_seed, threshold, fp_seed)
    w_ends, w_fps, w_n = orc.cdc(ts.stream_off, ts.tokens, gear_seed, threshold, fp_seed)
    assert status == kv.KV_OK
    assert n == w_n
    assert np.array_equal(ends, w_ends)
    assert np.array_equal(fps, w_fps)
    return n


# lengths around the 32-token runs, the 64-token window and the 8192-token
# tiles of the kernels, with empty streams between them
RAGGED = [0, 1, 31, 32, 33, 63, 64, 65, 0, 0, 127, 8191, 8192, 8193, 100, 20000, 1, 0]


@pytest.mark.parametrize("log_len", [4, 8, 12])
def test_cdc_matches_oracle_on_ragged_streams(orc, log_len):
    ts = synth.token_streams(21 + log_len, RAGGED, shared_segments=3, segment_lo=50,
                             segment_hi=3000)
    n = _check(orc, ts, 0x1234, 1 << (64 - log_len), fp_seed=77)
    assert n > sum(1 for x in RAGGED if x)


def test_cdc_many_streams_long_and_short(orc):
    rng = np.random.default_rng(5)
    lengths = rng.integers(0, 3000, 700).tolist() + [300000, 70000]
    ts = synth.token_streams(31, lengths, shared_segments=16)
    _check(orc, ts, 99, 1 << 56)


def test_cdc_threshold_extremes(orc):
    ts = synth.token_streams(41, [5000, 0, 77, 12000])
    assert _check(orc, ts, 1, 0) == 3            # stream ends only
    assert _check(orc, ts, 1, M64) == len(ts.tokens)   # (nearly) every token


def test_cdc_repeated_content_gives_repeated_fingerprints(orc):
    # one segment pasted into many streams at different offsets: past its
    # first 64 tokens its chunks (boundaries and fingerprints) recur
    seg = synth.token_streams(51, [6000]).tokens
    parts, rng = [], np.random.default_rng(9)
    for _ in range(6):
        parts.append(synth.token_streams(int(rng.integers(1000)), [int(rng.integers(64, 3000))]).tokens)
        parts.append(seg)
    lengths = [len(p) for p in parts]
    ts = synth.TokenStreams(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
                            np.concatenate(parts))
    status, n, ends, fps = _run(ts, 3, 1 << 58)
    w_ends, w_fps, _ = orc.cdc(ts.stream_off, ts.tokens, 3, 1 << 58)
    assert status == kv.KV_OK and np.array_equal(ends, w_ends) and np.array_equal(fps, w_fps)
    values, counts = np.unique(fps, return_counts=True)
    assert counts.max() >= 6


def test_cdc_capacity_is_reported_and_prefix_kept(orc):
    ts = synth.token_streams(61, [4000, 4000])
    w_ends, w_fps, w_n = orc.cdc(ts.stream_off, ts.tokens, 7, 1 << 58)
    cap = w_n // 2
    status, n, ends, fps = _run(ts, 7, 1 << 58, max_chunks=cap)
    assert status == kv.KV_ERR_CAPACITY and n == w_n
    assert np.array_equal(ends, w_ends[:cap]) and np.array_equal(fps, w_fps[:cap])


def test_cdc_offsets_that_miss_the_token_count_are_reported(orc):
    ts = synth.token_streams(71, [500, 500])
    bad = synth.TokenStreams(np.array([0, 500, 900], dtype=np.int64), ts.tokens)
    status, _, _, _ = _run(bad, 7, 1 << 58)
    assert status == kv.KV_ERR_OUT_OF_RANGE


def test_cdc_empty_input():
    ts = synth.TokenStreams(np.zeros(3, dtype=np.int64), np.zeros(0, dtype=np.int32))
    status, n, _, _ = _run(ts, 1, 1 << 58)
    assert status == kv.KV_OK and n == 0


def test_fixed_window_fingerprints(orc):
    # the fallback S1: consecutive 128-token windows (the last one shorter)
    ts = synth.token_streams(81, [100000 + 77])
    total = len(ts.tokens)
    starts = np.arange(0, total, 128, dtype=np.int64)
    ends = np.minimum(starts + 128, total).astype(np.int64)
    want = orc.fingerprint(starts, ends, ts.tokens, 5)
    out = torch.zeros(len(starts), dtype=torch.int64, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    kv.kv_fingerprint(len(starts), torch.from_numpy(starts).cuda(), torch.from_numpy(ends).cuda(),
                      total, torch.from_numpy(ts.tokens).cuda(), 5, out, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert np.array_equal(out.cpu().numpy().view(np.uint64), want)
    assert kv.kv_last_launch_count() == 1
