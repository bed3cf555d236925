"""Benchmark of the KV relocation / splice / patch path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--check]

With no --workload, every configured workload prints one JSON line (rank 0),
in this order, the headline last:
  splice-mla-4k       Leyline splice on one MLA layer of 4096 tokens,
                      [1024, 2048) -> 16-row stub (L2-resident);
  splice-mla-128k     Leyline AMORTIZE at 128K context: 61 layers, 8 sequences
                      of 131072 tokens, 4 successive directives each;
  relocate-gqa-patch  Kamera GQA relocation (32 layers, 8 x 128 K and V) with
                      a fused rank-16 patch on K and V;
  sweep-mla           MLA relocation over chunk lengths 16..4096 x δ in
                      {±1, ±1000, ±100000}, the splice with Δ = δ and the
                      standalone rank-8 patch (one summary line);
  relocate-mla        the headline: Irminsul-style relocation with a
                      DeepSeek-V3-shaped MLA cache -- 61 layers, rows of c_KV
                      512 + k_pe 64 bf16, 64-token blocks, 32 requests each
                      assembling 16 chunks (U[256, 2048] tokens) from a
                      256-chunk registry, δ U[-32768, 32768]; one step = one
                      kv_relocate call (δ-table + relocation kernels).
Other workloads (--workload): relocate-mla-patch, splice-mla-128k-composed,
splice-mla-128k-remap (and -split), window-gqa, families, cdc-tokens.

``value`` is the workload's metric for the whole job (relocated KV tokens/s
over all layers); ``roofline`` gives the dominant kernel's achieved HBM
bandwidth (algorithmic bytes per launch / CUDA-event time on its stream)
against the measured copy peak; ``e2e`` is the same metric through the C-ABI
call with the step's inputs copied from pinned host memory and the status
word read back every step; ``cpu_baseline`` is the fp64 oracle timed on
bounded samples of the same recipe on every host core and on one core.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

MLA_ROW = 576           # c_KV 512 + k_pe 64 (bf16)
MLA_ROW_BYTES = 1152
GQA_ROW_BYTES = 2048    # K or V: 8 heads x 128 x bf16
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth (context for the measured fraction)


def add_nominal(out: dict) -> dict:
    """Beside the fraction of the measured copy bandwidth, the fraction of
    the nominal HBM3e bandwidth."""
    r = out.get("roofline") or {}
    if r.get("bound") == "hbm" and r.get("unit") == "GB/s" and "achieved" in r:
        r["nominal_peak"] = NOMINAL_HBM_GBS
        r["frac_of_nominal"] = r["achieved"] / NOMINAL_HBM_GBS
    return out


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Sources that decide a workload's row-moving kernels (their device code and
# launch parameters): a recorded DRAM traffic figure is used only while these
# files are unchanged.  kv_api.cu is included where it plans the launch (splice
# tiles, remapping); it only forwards arguments for relocation and chunking.
_DEVICE_SOURCES = ("kv_device.cuh", "kv_tiles.cuh", "kv_internal.h")
KERNEL_SOURCES = {
    "relocate_mla": ("kv_relocate.cu",) + _DEVICE_SOURCES,
    "splice_mla_128k": ("kv_splice.cu", "kv_api.cu") + _DEVICE_SOURCES,
    "relocate_gqa_patch": ("kv_patch_tc.cu",) + _DEVICE_SOURCES,
    "relocate_mla_patch": ("kv_patch_tc.cu",) + _DEVICE_SOURCES,
    "splice_mla_128k_composed": ("kv_splice.cu", "kv_api.cu") + _DEVICE_SOURCES,
    "splice_mla_128k_remap": ("kv_splice.cu", "kv_api.cu") + _DEVICE_SOURCES,
    "window_gqa": ("kv_splice.cu", "kv_patch_tc.cu", "kv_api.cu") + _DEVICE_SOURCES,
    "cdc_tokens": ("kv_cdc.cu", "kv_device.cuh", "kv_internal.h"),
    "families": ("kv_relocate.cu",) + _DEVICE_SOURCES,
    "sweep_mla": ("kv_relocate.cu",) + _DEVICE_SOURCES,
}


def kernel_sources_hash(workload: str) -> str:
    """sha256 (16 hex digits) of the sources that build `workload`'s kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "position_independent_mla_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[workload]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary (captured on the workload's small case and scaled by the ratio of
    algorithmic bytes), or None when that summary was taken on other kernel
    sources."""
    path = os.path.join(ROOT, "profiles", f"{workload}_traffic.txt")
    try:
        kv = dict(line.strip().split("=", 1) for line in open(path)
                  if "=" in line and not line.startswith("#"))
    except OSError:
        return None
    if kv.get("kernel_sources_sha256_16") != kernel_sources_hash(workload):
        return None
    # the figure is scaled from a small case; absent where the small case's
    # traffic does not grow in proportion to the workload
    return float(kv["dram_bytes_per_launch"]) if "dram_bytes_per_launch" in kv else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.path = None

    def start(self):
        try:
            ident = str(torch.cuda.get_device_properties(self.device).uuid)
            ident = ident if ident.startswith("GPU-") else "GPU-" + ident
        except Exception:
            ident = str(self.device)
        self.path = f"/tmp/kvreloc_clocks_{os.getpid()}.csv"
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", ident], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def ulp_stats(got: np.ndarray, want: np.ndarray) -> dict:
    """Compare bf16 bit patterns as the parity tests do: exact, within 1 ulp,
    and beyond (more than 1 ulp AND more than 1e-6 apart); NaN must meet NaN."""
    g, w = got.astype(np.int64).ravel(), want.astype(np.int64).ravel()
    og = np.where(g & 0x8000, 0x8000 - (g & 0x7FFF), 0x8000 + g)
    ow = np.where(w & 0x8000, 0x8000 - (w & 0x7FFF), 0x8000 + w)
    gf = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(gf) | np.isnan(wf)
    dist = np.abs(og - ow)
    with np.errstate(invalid="ignore"):
        far = (dist > 1) & ~(np.abs(gf - wf) <= 1e-6)
    far = np.where(nan, np.isnan(gf) != np.isnan(wf), far)
    return {"exact": int((dist == 0).sum()), "one_ulp": int((dist == 1).sum()),
            "beyond": int(far.sum()), "values": int(dist.size)}


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def fill_normal_(t: torch.Tensor, seed: int) -> None:
    """Fill a bf16 [L][...] device tensor with N(0,1) draws, one layer at a time."""
    g = torch.Generator(device=t.device)
    for l in range(t.shape[0]):
        g.manual_seed(seed * 1000 + l)
        t[l].copy_(torch.randn(t[l].shape, generator=g, device=t.device, dtype=torch.float32))


# ---------------------------------------------------------------------------
# Workload: Irminsul relocation, MLA, 61 layers (default)
# ---------------------------------------------------------------------------

RELOC_MLA = dict(layers=61, num_reqs=32, chunks_per_req=16, len_lo=256, len_hi=2048,
                 delta_lo=-32768, delta_hi=32768, n_pool_chunks=256, base_hi=32768, base=10000.0)


def build_relocate_mla(rank: int, device: str = "cuda", cfg=RELOC_MLA):
    import position_independent_mla_gb300 as kv

    c = cfg
    wl = synth.relocate_workload(1002 + 100 * rank, num_reqs=c["num_reqs"],
                                 chunks_per_req=c["chunks_per_req"], len_lo=c["len_lo"],
                                 len_hi=c["len_hi"], delta_lo=c["delta_lo"],
                                 delta_hi=c["delta_hi"], n_pool_chunks=c["n_pool_chunks"],
                                 base_hi=c["base_hi"])
    L = c["layers"]
    src = torch.empty((L, wl.src_slots_total, MLA_ROW), dtype=torch.bfloat16, device=device)
    fill_normal_(src, 1002 + 100 * rank)
    dst = torch.zeros((L, wl.dst_slots_total, MLA_ROW), dtype=torch.bfloat16, device=device)
    sd = kv.pool_desc(src[..., :512], src[..., 512:], 64, 1, c["base"])
    dd = kv.pool_desc(dst[..., :512], dst[..., 512:], 64, 1, c["base"])
    host = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).pin_memory()
            for k in ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta",
                      "block_tables")}
    dev = {k: v.to(device) for k, v in host.items()}
    ws = kv.workspace(dd, wl.total_tokens, wl.num_chunks, device=device)
    return dict(wl=wl, src=src, dst=dst, sd=sd, dd=dd, host=host, dev=dev, ws=ws, L=L, cfg=c)


def relocate_call(st, dev=None, stream=None):
    import position_independent_mla_gb300 as kv

    wl, d = st["wl"], dev if dev is not None else st["dev"]
    kv.kv_relocate(st["sd"], st["dd"], wl.num_chunks, wl.total_tokens, d["tok_off"],
                   d["src_slots"], d["chunk_req"], d["chunk_dst_pos"], d["delta"],
                   d["block_tables"], wl.block_tables.shape[0], wl.block_tables.shape[1], None,
                   st["ws"], stream=stream)
    return kv.kv_last_launch_count()


def check_relocate_sample(st, orc, n_rows: int = 3000, seed: int = 7) -> dict:
    """Sampled parity at full size: random (token, layer) rows of the last
    relocation, each compared with the oracle's rotation of its source row."""
    wl, L = st["wl"], st["L"]
    rng = np.random.default_rng(seed)
    toks = rng.integers(0, wl.total_tokens, n_rows)
    lays = rng.integers(0, L, n_rows)
    chunk = np.searchsorted(wl.tok_off, toks, side="right") - 1
    pos = wl.chunk_dst_pos[chunk] + (toks - wl.tok_off[chunk])
    dslot = wl.block_tables[wl.chunk_req[chunk], pos // 64].astype(np.int64) * 64 + pos % 64
    sslot = wl.src_slots[toks].astype(np.int64)
    li = torch.from_numpy(lays).cuda()
    srows = st["src"][li, torch.from_numpy(sslot).cuda()].cpu()
    drows = st["dst"][li, torch.from_numpy(dslot).cuda()].cpu()
    sb, db = synth.bits(srows), synth.bits(drows)
    copy_bad = int((sb[:, :512] != db[:, :512]).any(axis=1).sum())
    want = np.stack([orc.rotate_bf16(sb[i, 512:], int(wl.delta[chunk[i]]), st["cfg"]["base"])
                     for i in range(n_rows)])
    r = ulp_stats(db[:, 512:], want)
    return {"rows": n_rows, "copy_rows_differing": copy_bad, "rot_exact": r["exact"],
            "rot_one_ulp": r["one_ulp"], "rot_beyond": r["beyond"]}


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle, as it stands, on bounded samples of each
# workload's recipe, timed on one host core and on every host core at once
# (one spawned process per core, each on its own independent sample; the
# oracle's arithmetic is unchanged)
# ---------------------------------------------------------------------------

def _mla_pool(O, L, slots, seed, base=10000.0):
    return O.Pool(synth.bits(synth.bf16_normal((L, slots, 512), seed)).copy(),
                  synth.bits(synth.bf16_normal((L, slots, 64), seed + 1)).copy(), 64, 1, 64, base)


def oracle_sample(kind: str, n: int, seed: int):
    """One bounded oracle sample of workload `kind` (size parameter `n`):
    returns (call, units, what) -- `call()` runs the oracle once, `units` is
    the metric's units one call yields (rows or tokens moved, all layers),
    `what` describes the sample."""
    import oracle as O

    orc = O.get()
    if kind in ("relocate-mla", "sweep-mla"):
        c = RELOC_MLA
        if kind == "relocate-mla":   # one chunk of n tokens, the headline's δ range
            wl = synth.relocate_workload(seed, num_reqs=1, chunks_per_req=1, len_lo=n, len_hi=n,
                                         delta_lo=c["delta_lo"], delta_hi=c["delta_hi"],
                                         n_pool_chunks=1, base_hi=63)
            what = f"one {n}-token chunk, 61 layers"
        else:                        # 8n short chunks over the sweep's range of shifts
            wl = synth.relocate_workload(seed, num_reqs=1, chunks_per_req=8 * n, len_lo=16,
                                         len_hi=256, delta_lo=-100000, delta_hi=100000,
                                         n_pool_chunks=8 * n, base_hi=63)
            what = f"one request of {8 * n} chunks of U[16,256] tokens, 61 layers"
        L = c["layers"]
        src = _mla_pool(O, L, wl.src_slots_total, seed)
        dst = O.Pool(np.zeros((L, wl.dst_slots_total, 512), np.uint16),
                     np.zeros((L, wl.dst_slots_total, 64), np.uint16), 64, 1, 64, c["base"])

        def call():
            assert orc.relocate(src, dst, wl.tok_off, wl.src_slots, wl.chunk_req,
                                wl.chunk_dst_pos, wl.delta, wl.block_tables) == O.OK
        return call, wl.total_tokens, what
    if kind == "relocate-gqa-patch":   # n chunks of 576 tokens, rank-16 patch on K and V
        c = RELOC_GQA
        wl = synth.relocate_workload(seed, num_reqs=1, chunks_per_req=n, len_lo=c["chunk_len"],
                                     len_hi=c["chunk_len"], delta_lo=c["delta_lo"],
                                     delta_hi=c["delta_hi"], n_pool_chunks=n, base_hi=63)
        L, m = c["layers"], c["rank"]
        src = O.Pool(synth.bits(synth.bf16_normal((L, wl.src_slots_total, 1024), seed)).copy(),
                     synth.bits(synth.bf16_normal((L, wl.src_slots_total, 1024), seed + 1)).copy(),
                     64, 8, 128, c["base"])
        dst = O.Pool(np.zeros((L, wl.dst_slots_total, 1024), np.uint16),
                     np.zeros((L, wl.dst_slots_total, 1024), np.uint16), 64, 8, 128, c["base"])
        u = [synth.f32_normal((L, wl.total_tokens, m), seed + 2 + i, std=c["std"]).numpy()
             for i in range(2)]
        v = [synth.f32_normal((L, wl.num_chunks, 1024, m), seed + 4 + i, std=c["std"]).numpy()
             for i in range(2)]
        patch = O.Patch(m, u, v)

        def call():
            assert orc.relocate(src, dst, wl.tok_off, wl.src_slots, wl.chunk_req,
                                wl.chunk_dst_pos, wl.delta, wl.block_tables, patch) == O.OK
        return call, wl.total_tokens, f"{n} chunk(s) of 576 tokens, 32 layers, rank-16 patch"
    if kind in ("splice-mla-128k", "splice-mla-4k"):
        if kind == "splice-mla-4k":    # the whole configured case: 1 layer, 4096 tokens
            c = SPLICE_4K
            L, seq = 1, c["seq_len"]
            s0, s1, nr = c["s_start"], c["s_end"], c["stub"]
            what = "the whole case (1 layer, 4096 tokens, [1024,2048) -> 16 rows)"
        else:                          # one n-token sequence, one directive, all 61 layers
            c = SPLICE_128K
            L, seq = c["layers"], n
            d = synth.random_directives(seed, [seq], seq // 16, seq // 4, c["stub_lo"],
                                        c["stub_hi"])
            s0, s1, nr = int(d.s_start[0]), int(d.s_end[0]), int(d.stub_len[0])
            what = (f"one {seq}-token sequence, 61 layers, one directive removing {s1 - s0} "
                    f"tokens for a {nr}-row stub")
        ss = synth.splice_seqs(seed, [seq], (seq + 63) // 64)
        pool = _mla_pool(O, L, ss.num_slots, seed, c["base"])
        sc = synth.bits(synth.bf16_normal((L, nr, 512), seed + 2)).copy()
        sr = synth.bits(synth.bf16_normal((L, nr, 64), seed + 3)).copy()
        moved = (seq - s1) + nr

        def call():
            lens = np.array([seq], np.int32)
            assert orc.splice(pool, ss.block_tables, lens, [s0], [s1], [nr], sc, sr) == O.OK
        return call, moved, what
    raise ValueError(kind)


_CORE_BARRIER = None


def _core_init(barrier):
    global _CORE_BARRIER
    _CORE_BARRIER = barrier
    torch.set_num_threads(1)  # one core per process, also while drawing the sample


def _core_task(kind: str, n: int, seed: int, min_seconds: float):
    """One core's share: build its sample (untimed), wait for every core, then
    run the oracle on it until `min_seconds` have passed.  Returns (units,
    start, end, what) on the system-wide monotonic clock."""
    call, units, what = oracle_sample(kind, n, seed)
    if _CORE_BARRIER is not None:
        _CORE_BARRIER.wait(timeout=600)
    t0 = time.monotonic()
    reps = 0
    while reps == 0 or time.monotonic() - t0 < min_seconds:
        call()
        reps += 1
    return units * reps, t0, time.monotonic(), what


class OracleCores:
    """A pool of spawned processes, one per host core, that run the oracle
    side by side; each round starts all of them together behind a barrier."""

    def __init__(self, n: int | None = None):
        import concurrent.futures as cf
        import multiprocessing as mp

        self.n = n or os.cpu_count() or 1
        ctx = mp.get_context("spawn")
        self.pool = cf.ProcessPoolExecutor(self.n, mp_context=ctx, initializer=_core_init,
                                           initargs=(ctx.Barrier(self.n),))

    def run(self, kind: str, n: int, seed: int, min_seconds: float = 0.0):
        """Every core runs its own sample of `kind`; returns (units, seconds,
        what) with seconds from the first start to the last end."""
        futs = [self.pool.submit(_core_task, kind, n, seed + 7919 * i, min_seconds)
                for i in range(self.n)]
        res = [f.result() for f in futs]
        return sum(r[0] for r in res), max(r[2] for r in res) - min(r[1] for r in res), res[0][3]

    def close(self):
        self.pool.shutdown()


def cpu_model() -> str:
    try:
        for line in subprocess.run(["lscpu"], capture_output=True, text=True).stdout.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


# Sample size per core and per single-thread run of each workload's oracle
# baseline, and the seconds each is timed for.
CPU_SAMPLES = {"relocate-mla": (512, 4096, 10.0), "sweep-mla": (1, 2, 4.0),
               "relocate-gqa-patch": (1, 1, 4.0), "splice-mla-128k": (4096, 8192, 4.0),
               "splice-mla-4k": (0, 0, 4.0)}


def cpu_baseline(kind: str, unit: str, cores: "OracleCores | None" = None) -> dict:
    """The oracle on every host core at once and on one core, on bounded
    samples of `kind`'s recipe."""
    n_all, n_one, secs = CPU_SAMPLES[kind]
    own = cores is None
    if own:
        cores = OracleCores()
    try:
        cores.run("splice-mla-4k", 0, 1, 0.0)   # spawn and import everywhere, untimed
        units, dt, what = cores.run(kind, n_all, 9001, secs)
    finally:
        if own:
            cores.close()
    u1, t0, t1, what1 = _core_task(kind, n_one, 4242, secs)
    return {"value": units / dt, "unit": unit, "cores": cores.n, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{cores.n} processes side by side, each on its own sample ({what}) "
                      f"for {dt:.1f} s",
            "single_thread": {"value": u1 / (t1 - t0), "unit": unit, "cores": 1,
                              "sample": f"{what1}, repeated for {t1 - t0:.1f} s"}}


# A small case of the same kernel for ncu captures (a few GB on the device).
RELOC_MLA_SMALL = dict(RELOC_MLA, num_reqs=2, n_pool_chunks=16)


def run_relocate_mla(args, rank, world, local):
    import position_independent_mla_gb300 as kv

    st = build_relocate_mla(rank, cfg=RELOC_MLA_SMALL if args.small else RELOC_MLA)
    wl, L = st["wl"], st["L"]
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        relocate_call(st)
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for a, b in ev:  # torch creates the CUDA event on its first record()
        a.record()
        b.record()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    launches = 0
    t_start.record()
    for i in range(K):
        kv.kv_set_kernel_events(*ev[i])
        launches += relocate_call(st)
    t_stop.record()
    torch.cuda.synchronize()
    barrier(world)
    kv.kv_set_kernel_events(None, None)
    step_ms = t_start.elapsed_time(t_stop) / K
    kern_ms = sum(a.elapsed_time(b) for a, b in ev) / K

    # end to end through the C ABI: host index arrays -> device, call, status back
    host, dev = st["host"], st["dev"]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(K):
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        relocate_call(st, dev)
        status = kv.kv_get_device_status(st["ws"], stream)
        assert status == kv.KV_OK, kv.status_string(status)
    e2e_s = time.perf_counter() - t0
    barrier(world)
    clk = clocks.stop()

    step_ms = max_over_ranks(step_ms, world)
    kern_ms_max = max_over_ranks(kern_ms, world)
    e2e_s = max_over_ranks(e2e_s, world)
    tokens = wl.total_tokens
    total_tokens = tokens * world  # weak scaling: every rank relocates its own batch

    check = None
    if args.check and rank == 0:
        import oracle as O
        check = check_relocate_sample(st, O.get())

    bytes_per_launch = tokens * (L * 2 * MLA_ROW_BYTES + 4)
    peak, peak_kind = hbm_peak()
    achieved = bytes_per_launch / (kern_ms * 1e-3) / 1e9
    traffic = recorded_traffic("relocate_mla")
    out = {
        "metric": "relocated KV tokens/s (all layers)",
        "value": total_tokens / (step_ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": "irminsul-relocate-mla: 61 layers, c_KV 512 + k_pe 64 bf16, "
                               "64-token blocks, 32 requests x 16 chunks of U[256,2048] tokens "
                               "from a 256-chunk registry, delta U[-32768,32768]",
                   "tokens_per_step_per_gpu": tokens, "layers": L, "chunks": wl.num_chunks,
                   "parallelism": f"replicas x{world} (independent batches)",
                   "l2": "inputs larger than L2 (%.1f GB moved per step)" % (
                       bytes_per_launch / 1e9),
                   "math": "fp64 angles, compensated fp32 rotation, one bf16 rounding"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic, "kernel": "relocate_kernel<MLA>",
                     "kernel_ms": kern_ms, "kernel_ms_max_over_ranks": kern_ms_max,
                     "algorithmic_bytes_per_launch": bytes_per_launch},
        "e2e": {"value": total_tokens * K / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "clocks": clk,
        "gpu_launches": launches,
    }
    if check is not None:
        out["parity_sample"] = check
    return out


def check_reloc_mla_patch_sample(st, u, v, m, orc, n_rows: int = 300, seed: int = 17) -> dict:
    """Sampled parity at full size for the patched MLA relocation: random
    (token, layer) rows, each checked against the oracle's fused relocation +
    patch on a one-token problem built from that row's source values and its
    U / V factors (one 576-wide factor pair split at column 512)."""
    import oracle as O

    wl, L, base = st["wl"], st["L"], st["cfg"]["base"]
    rng = np.random.default_rng(seed)
    out = {"copy_beyond": 0, "rot_beyond": 0, "exact": 0, "one_ulp": 0, "values": 0}
    for _ in range(n_rows):
        t = int(rng.integers(wl.total_tokens))
        l = int(rng.integers(L))
        c = int(np.searchsorted(wl.tok_off, t, side="right") - 1)
        pos = int(wl.chunk_dst_pos[c]) + t - int(wl.tok_off[c])
        ds = int(wl.block_tables[wl.chunk_req[c], pos // 64]) * 64 + pos % 64
        row = synth.bits(st["src"][l, int(wl.src_slots[t])].cpu())
        sc, sr = np.zeros((1, 64, 512), np.uint16), np.zeros((1, 64, 64), np.uint16)
        sc[0, 0], sr[0, 0] = row[:512], row[512:]
        src = O.Pool(sc, sr, 64, 1, 64, base)
        dst = O.Pool(np.zeros((1, 64, 512), np.uint16), np.zeros((1, 64, 64), np.uint16), 64, 1,
                     64, base)
        ut = u[l, t].cpu().numpy().reshape(1, 1, m)
        vc = v[l, c].cpu().numpy().reshape(1, 1, 576, m)
        assert orc.relocate(src, dst, [0, 1], [0], [0], [0], [int(wl.delta[c])], [[0]],
                            O.Patch(m, [ut, ut], [vc[:, :, :512], vc[:, :, 512:]])) == O.OK
        got = synth.bits(st["dst"][l, ds].cpu())
        for g, want, key in ((got[:512], dst.copy[0, 0], "copy_beyond"),
                             (got[512:], dst.rot[0, 0], "rot_beyond")):
            r = ulp_stats(g, want)
            out[key] += r["beyond"]
            out["exact"] += r["exact"]
            out["one_ulp"] += r["one_ulp"]
            out["values"] += r["values"]
    out["rows"] = n_rows
    return out


def run_relocate_mla_patch(args, rank, world, local):
    """The headline relocation with Kamera's rank-8 patch fused: one factor
    pair over the 576-wide MLA row (c_KV and k_pe both patched), fp32
    factors N(0, 0.02^2) per (token, layer) for U and (chunk, layer) for V."""
    import position_independent_mla_gb300 as kv

    st = build_relocate_mla(rank, cfg=RELOC_MLA_SMALL if args.small else RELOC_MLA)
    wl, L, m = st["wl"], st["L"], 8
    g = torch.Generator(device="cuda")
    g.manual_seed(6006 + 100 * rank)
    u = torch.randn((L, wl.total_tokens, m), generator=g, device="cuda").mul_(0.02)
    v = torch.randn((L, wl.num_chunks, 576, m), generator=g, device="cuda").mul_(0.02)
    patch = kv.patch_desc(m, [u, u], [v[:, :, :512], v[:, :, 512:]])
    d = st["dev"]

    def call():
        kv.kv_relocate(st["sd"], st["dd"], wl.num_chunks, wl.total_tokens, d["tok_off"],
                       d["src_slots"], d["chunk_req"], d["chunk_dst_pos"], d["delta"],
                       d["block_tables"], wl.block_tables.shape[0], wl.block_tables.shape[1],
                       patch, st["ws"])
        return kv.kv_last_launch_count()

    for _ in range(args.warmup):
        call()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for a, b in ev:
        a.record()
        b.record()
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    launches = 0
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record()
    for i in range(K):
        kv.kv_set_kernel_events(*ev[i])
        launches += call()
    t_stop.record()
    torch.cuda.synchronize()
    kv.kv_set_kernel_events(None, None)
    clk = clocks.stop()
    assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
    step_ms = t_start.elapsed_time(t_stop) / K
    kern_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    T = wl.total_tokens
    bytes_launch = T * (L * 2 * MLA_ROW_BYTES + 4) + T * L * m * 4 + wl.num_chunks * L * 576 * m * 4
    peak, peak_kind = hbm_peak()
    achieved = bytes_launch / (kern_ms * 1e-3) / 1e9
    out = {
        "metric": "relocated KV tokens/s (all layers)", "value": T * world / (step_ms * 1e-3),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": "irminsul-relocate-mla + fused rank-8 patch over the 576-wide row",
                   "tokens_per_step_per_gpu": T, "layers": L},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic("relocate_mla_patch"),
                     "kernel": "patch_tc_kernel (c_KV: 256-column slices; k_pe: 64)",
                     "kernel_ms": kern_ms, "algorithmic_bytes_per_launch": bytes_launch},
        "clocks": clk, "gpu_launches": launches,
    }
    if args.check and rank == 0:
        import oracle as O
        out["parity_sample"] = check_reloc_mla_patch_sample(st, u, v, m, O.get())
    return out


# ---------------------------------------------------------------------------
# Workload: Leyline AMORTIZE at 128K context, MLA, 61 layers
# ---------------------------------------------------------------------------

SPLICE_128K = dict(layers=61, num_seqs=8, seq_len=131072, rounds=4, span_lo=8192,
                   span_hi=32768, stub_lo=8, stub_hi=64, base=10000.0)
# A small case of the same kernel for ncu captures (~2.3 GB pool).
SPLICE_128K_SMALL = dict(SPLICE_128K, num_seqs=1, seq_len=32768, span_lo=2048, span_hi=8192)


class SplitPool:
    """An MLA pool stored as two tensors, c_KV [L][slots][512] and k_pe
    [L][slots][64]; indexing returns the joined 576-wide rows."""

    def __init__(self, c: torch.Tensor, r: torch.Tensor):
        self.c, self.r = c, r

    def __getitem__(self, idx):
        return torch.cat([self.c[idx], self.r[idx]], -1)

    def copy_(self, other: "SplitPool"):
        self.c.copy_(other.c)
        self.r.copy_(other.r)
        return self

    def clone(self) -> "SplitPool":
        return SplitPool(self.c.clone(), self.r.clone())


def build_splice(rank: int, cfg, device: str = "cuda", aligned: bool = False,
                 split: bool = False):
    """The 128K-context splice workload.  `split`: the pool as separate c_KV
    and k_pe tensors instead of one [L][slots][576] tensor."""
    import position_independent_mla_gb300 as kv

    c = cfg
    L, S, n = c["layers"], c["num_seqs"], c["seq_len"]
    max_blocks = (n + 63) // 64          # spans (>= 8K) outgrow stubs: sequences shrink
    ss = synth.splice_seqs(3003 + 100 * rank, [n] * S, max_blocks)
    if split:
        pool = SplitPool(torch.empty((L, ss.num_slots, 512), dtype=torch.bfloat16, device=device),
                         torch.empty((L, ss.num_slots, 64), dtype=torch.bfloat16, device=device))
        fill_normal_(pool.c, 3003 + 100 * rank)
        fill_normal_(pool.r, 3053 + 100 * rank)
        desc = kv.pool_desc(pool.c, pool.r, 64, 1, c["base"])
    else:
        pool = torch.empty((L, ss.num_slots, MLA_ROW), dtype=torch.bfloat16, device=device)
        fill_normal_(pool, 3003 + 100 * rank)
        desc = kv.pool_desc(pool[..., :512], pool[..., 512:], 64, 1, c["base"])
    pristine = pool.clone()
    lens = ss.seq_lens.copy()
    rounds = []
    for r in range(c["rounds"]):
        if aligned:   # whole blocks: U[1, 4] stub blocks
            d = synth.random_aligned_directives(3100 + 100 * rank + r, lens, c["span_lo"],
                                                c["span_hi"], 1, 4)
        else:
            d = synth.random_directives(3100 + 100 * rank + r, lens, c["span_lo"], c["span_hi"],
                                        c["stub_lo"], c["stub_hi"])
        tot = int(d.stub_len.sum())
        stub_c = torch.empty((L, tot, 512), dtype=torch.bfloat16, device=device)
        stub_r = torch.empty((L, tot, 64), dtype=torch.bfloat16, device=device)
        fill_normal_(stub_c, 3200 + 100 * rank + r)
        fill_normal_(stub_r, 3300 + 100 * rank + r)
        moved = int(np.sum(lens - d.s_end)) + tot
        rounds.append(dict(d=d, stub_c=stub_c, stub_r=stub_r, lens_before=lens.copy(),
                           moved=moved, args=[torch.from_numpy(x.copy()) for x in
                                              (d.s_start, d.s_end, d.stub_len)]))
        lens = lens + d.stub_len - (d.s_end - d.s_start)
    ws = kv.workspace(desc, S * n, S, device=device)
    bt = torch.from_numpy(ss.block_tables).to(device)
    return dict(ss=ss, pool=pool, pristine=pristine, desc=desc, rounds=rounds, ws=ws, bt=bt,
                L=L, S=S, final_lens=lens, cfg=c, max_blocks=max_blocks)


def splice_step(st, stream=None, mode=None):
    """All directive rounds on the restored cache; returns kernels launched."""
    import position_independent_mla_gb300 as kv

    mode = kv.KV_AMORTIZE if mode is None else mode
    lens = torch.from_numpy(st["ss"].seq_lens.copy())
    launches = 0
    for rd in st["rounds"]:
        s0, s1, nr = rd["args"]
        kv.kv_splice(st["desc"], st["S"], st["bt"], st["max_blocks"], lens, s0, s1, nr,
                     rd["stub_c"], rd["stub_r"], mode, st["ws"], stream=stream)
        launches += kv.kv_last_launch_count()
    return launches, lens


def check_splice_sample(st, orc, n_rows: int = 2000, seed: int = 11,
                        composed: bool = False, final_bt=None) -> dict:
    """Sampled parity at full size: random (sequence, final position, layer)
    rows after all directive rounds, each traced back through the rounds to
    its origin (an original row or a stub row) and compared with the oracle's
    rotations applied round by round (one bf16 rounding per round) -- or, for
    the composed edit, one rotation by the summed shift (one rounding)."""
    rng = np.random.default_rng(seed)
    L, S, bt = st["L"], st["S"], st["ss"].block_tables
    base = st["cfg"]["base"]
    stub_off = []
    for rd in st["rounds"]:
        stub_off.append(np.concatenate([[0], np.cumsum(rd["d"].stub_len)[:-1]]))
    want_c, want_r, have_idx = [], [], []
    for _ in range(n_rows):
        q = int(rng.integers(S))
        if st["final_lens"][q] == 0:
            continue
        p = int(rng.integers(st["final_lens"][q]))
        l = int(rng.integers(L))
        p_final, rots, origin = p, [], None
        for r in reversed(range(len(st["rounds"]))):
            d = st["rounds"][r]["d"]
            a, b, nr = int(d.s_start[q]), int(d.s_end[q]), int(d.stub_len[q])
            if p < a:
                continue
            if p < a + nr:
                origin = ("stub", r, int(stub_off[r][q]) + p - a)
                break
            delta = nr - (b - a)
            rots.append(delta)
            p -= delta
        if origin is None:
            origin = ("pool", p)
        slot = lambda pos: int(bt[q, pos // 64]) * 64 + pos % 64
        fbt = bt if final_bt is None else final_bt   # the block table after the edit
        final_slot = int(fbt[q, p_final // 64]) * 64 + p_final % 64
        if origin[0] == "pool":
            row = st["pristine"][l, slot(origin[1])]
            oc, orr = row[:512], row[512:]
        else:
            rd = st["rounds"][origin[1]]
            oc, orr = rd["stub_c"][l, origin[2]], rd["stub_r"][l, origin[2]]
        oc_b, or_b = synth.bits(oc.cpu()), synth.bits(orr.cpu())
        if composed:
            if sum(rots) != 0:
                or_b = orc.rotate_bf16(or_b, sum(rots), base)
        else:
            for delta in reversed(rots):
                or_b = orc.rotate_bf16(or_b, delta, base)
        want_c.append(oc_b)
        want_r.append(or_b)
        have_idx.append((l, final_slot))
    li = torch.tensor([x[0] for x in have_idx], device="cuda")
    si = torch.tensor([x[1] for x in have_idx], device="cuda")
    got = synth.bits(st["pool"][li, si].cpu())
    wc, wr = np.stack(want_c), np.stack(want_r)
    copy_bad = int((got[:, :512] != wc).any(axis=1).sum())
    r = ulp_stats(got[:, 512:], wr)
    return {"rows": len(have_idx), "copy_rows_differing": copy_bad,
            "rot_exact": r["exact"], "rot_one_ulp": r["one_ulp"], "rot_beyond": r["beyond"]}


def run_splice_mla_128k(args, rank, world, local):
    import position_independent_mla_gb300 as kv

    cfg = SPLICE_128K_SMALL if args.small else SPLICE_128K
    st = build_splice(rank, cfg)
    L = st["L"]
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        st["pool"].copy_(st["pristine"])
        splice_step(st)
    torch.cuda.synchronize()
    K, R = args.steps, len(st["rounds"])
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    kern_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K * R)]
    for a, b in step_ev + kern_ev:
        a.record()
        b.record()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    launches = 0
    for k in range(K):
        st["pool"].copy_(st["pristine"])      # restore the cache: not timed
        step_ev[k][0].record()
        lens = torch.from_numpy(st["ss"].seq_lens.copy())
        for r, rd in enumerate(st["rounds"]):
            kv.kv_set_kernel_events(*kern_ev[k * R + r])
            s0, s1, nr = rd["args"]
            kv.kv_splice(st["desc"], st["S"], st["bt"], st["max_blocks"], lens, s0, s1, nr,
                         rd["stub_c"], rd["stub_r"], kv.KV_AMORTIZE, st["ws"])
            launches += kv.kv_last_launch_count()
        step_ev[k][1].record()
    torch.cuda.synchronize()
    barrier(world)
    kv.kv_set_kernel_events(None, None)
    assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
    step_ms = sum(a.elapsed_time(b) for a, b in step_ev) / K
    kern_ms = sum(a.elapsed_time(b) for a, b in kern_ev) / K

    # end to end: each step restores the cache (untimed), then times, per
    # round, the copy of the prefilled stub rows from pinned host memory, the
    # call (the directive arguments are host arrays by design) and a status
    # read-back
    host_stubs = [(rd["stub_c"].cpu().pin_memory(), rd["stub_r"].cpu().pin_memory())
                  for rd in st["rounds"]]
    stub_bytes = sum(a.numel() * 2 + b.numel() * 2 for a, b in host_stubs)
    e2e_s = 0.0
    for k in range(K):
        st["pool"].copy_(st["pristine"])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        lens = torch.from_numpy(st["ss"].seq_lens.copy())
        for rd, (hc, hr) in zip(st["rounds"], host_stubs):
            rd["stub_c"].copy_(hc, non_blocking=True)
            rd["stub_r"].copy_(hr, non_blocking=True)
            s0, s1, nr = rd["args"]
            kv.kv_splice(st["desc"], st["S"], st["bt"], st["max_blocks"], lens, s0, s1, nr,
                         rd["stub_c"], rd["stub_r"], kv.KV_AMORTIZE, st["ws"])
            assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
        e2e_s += time.perf_counter() - t0
    clk = clocks.stop()
    step_ms = max_over_ranks(step_ms, world)
    e2e_s = max_over_ranks(e2e_s, world)

    moved = sum(rd["moved"] for rd in st["rounds"])
    bytes_per_step = moved * L * 2 * MLA_ROW_BYTES
    peak, peak_kind = hbm_peak()
    achieved = bytes_per_step / (kern_ms * 1e-3) / 1e9
    out = {
        "metric": "relocated KV tokens/s (all layers)",
        "value": moved * world / (step_ms * 1e-3), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": f"leyline-splice-mla: {L} layers, {st['S']} sequences x "
                               f"{cfg['seq_len']} tokens, {R} successive directives each "
                               f"removing U[{cfg['span_lo']},{cfg['span_hi']}] tokens at a "
                               f"random offset for a U[{cfg['stub_lo']},{cfg['stub_hi']}]-row "
                               f"stub; in place",
                   "rows_moved_per_step_per_gpu": moved, "layers": L,
                   "parallelism": f"replicas x{world} (independent sequences)",
                   "l2": "inputs larger than L2 (%.1f GB moved per step); cache restored "
                         "from a pristine copy between steps, untimed" % (bytes_per_step / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic("splice_mla_128k"),
                     "kernel": "splice_kernel<MLA>", "kernel_ms": kern_ms,
                     "launches_per_step": R, "kernel_ms_per_launch": kern_ms / R,
                     "algorithmic_bytes_per_launch": bytes_per_step / R,
                     "algorithmic_bytes_per_step": bytes_per_step},
        "e2e": {"value": moved * world * K / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": stub_bytes + 12 * st["S"] * R,
                "d2h_bytes_per_step": 4 * R,
                "copies": "per round: the stub rows from pinned host memory; the directive "
                          "(3 int32 per sequence) goes by value in the launch"},
        "clocks": clk, "gpu_launches": launches,
    }
    if args.check and rank == 0:
        import oracle as O
        out["parity_sample"] = check_splice_sample(st, O.get())
    return out


def run_splice_mla_128k_remap(args, rank, world, local, split: bool = False):
    """The 128K-context workload with block-aligned directives (spans of
    U[8192, 32768] tokens rounded to whole blocks at block-aligned offsets,
    stubs of 1-4 blocks), applied with KV_AMORTIZE_REMAP: downstream rows stay
    in their blocks, the block-table rows are permuted and only the rotary
    part is rewritten.  Timed against KV_AMORTIZE on the same directives;
    before each step the cache and the block tables are restored, untimed.
    `split`: c_KV and k_pe in separate tensors, so the rotary part of
    consecutive slots is contiguous (128 B rows) instead of 128 B out of every
    1152 B row of a fused pool."""
    import position_independent_mla_gb300 as kv

    cfg = SPLICE_128K_SMALL if args.small else SPLICE_128K
    st = build_splice(rank, cfg, aligned=True, split=split)
    L, R, S, K, W = st["L"], len(st["rounds"]), st["S"], args.steps, args.warmup
    bt0 = st["bt"].clone()

    def restore():
        st["pool"].copy_(st["pristine"])
        st["bt"].copy_(bt0)

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    ms, kms, launches = _timed(lambda: splice_step(st, mode=kv.KV_AMORTIZE_REMAP)[0], K, W,
                               prep=restore)
    amortize_ms, _, _ = _timed(lambda: splice_step(st)[0], K, W, prep=restore)
    barrier(world)
    clk = clocks.stop()
    assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
    ms = max_over_ranks(ms, world)
    # rows whose rotary part is rewritten in place (downstream) and stub rows
    down = sum(int(np.sum(rd["lens_before"] - rd["d"].s_end)) for rd in st["rounds"])
    stub = sum(int(np.sum(rd["d"].stub_len)) for rd in st["rounds"])
    nbytes = down * L * 2 * 128 + stub * L * 2 * MLA_ROW_BYTES
    moved = down + stub
    peak, peak_kind = hbm_peak()
    out = {
        "metric": "relocated KV tokens/s (all layers)",
        "value": moved * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": f"leyline-splice-mla-remap: {L} layers, {S} sequences x "
                               f"{cfg['seq_len']} tokens, {R} block-aligned directives (spans of "
                               f"U[{cfg['span_lo']},{cfg['span_hi']}] tokens in whole blocks, "
                               "stubs of 1-4 blocks) applied by block-table remapping; pool "
                               + ("split: c_KV [L][slots][512] and k_pe [L][slots][64]" if split
                                  else "fused: [L][slots][576]"),
                   "rows_moved_per_step_per_gpu": moved, "downstream_rows": down,
                   "stub_rows": stub, "layers": L, "amortize_ms": amortize_ms,
                   "speedup_vs_amortize": amortize_ms / ms,
                   "parallelism": f"replicas x{world} (independent sequences)",
                   "l2": "inputs larger than L2 (%.1f GB moved per step); cache and block "
                         "tables restored before each step, untimed" % (nbytes / 1e9)},
        "roofline": {"bound": "hbm", "achieved": nbytes / (kms * 1e-3) / 1e9 if kms > 0 else None,
                     "peak": peak, "unit": "GB/s", "peak_kind": peak_kind,
                     "traffic": (None if split else recorded_traffic("splice_mla_128k_remap")),
                     "kernel": "remap_data_kernel<MLA> (whole step: 4 rounds)",
                     "kernel_ms_last_round": kms, "algorithmic_bytes_per_step": nbytes,
                     "frac": None},
        "e2e": None, "clocks": clk, "gpu_launches": launches,
    }
    out["roofline"]["frac"] = nbytes / (ms * 1e-3) / 1e9 / peak   # whole step, all rounds
    out["roofline"]["achieved"] = nbytes / (ms * 1e-3) / 1e9
    if args.check and rank == 0:
        import oracle as O
        restore()
        splice_step(st, mode=kv.KV_AMORTIZE_REMAP)
        out["parity_sample"] = check_splice_sample(st, O.get(), final_bt=st["bt"].cpu().numpy())
    return out


def run_splice_mla_128k_composed(args, rank, world, local):
    """The 128K-context workload's directive rounds applied to each sequence as
    ONE composed edit (every row moved once, turned by its total shift,
    rounded once), timed against the successive kv_splice calls on the same
    directives.  Each timed call follows an untimed restore of the cache."""
    import position_independent_mla_gb300 as kv

    cfg = SPLICE_128K_SMALL if args.small else SPLICE_128K
    st = build_splice(rank, cfg)
    L, R, S, K, W = st["L"], len(st["rounds"]), st["S"], args.steps, args.warmup
    s0, s1, nr = (torch.stack([rd["args"][j] for rd in st["rounds"]]).contiguous()
                  for j in range(3))
    stub_c = torch.cat([rd["stub_c"] for rd in st["rounds"]], dim=1).contiguous()
    stub_r = torch.cat([rd["stub_r"] for rd in st["rounds"]], dim=1).contiguous()
    lens0 = st["ss"].seq_lens
    tl = torch.from_numpy(lens0.copy())
    ws = torch.empty(kv.kv_splice_composed_workspace_size(st["desc"], tl, s0, s1, nr),
                     dtype=torch.uint8, device="cuda")
    _, tiles, deltas = kv.kv_splice_composed_plan(st["desc"], tl, s0, s1, nr)
    rows = sum(t["n"] for t in tiles)
    restore = lambda: st["pool"].copy_(st["pristine"])

    def call():
        lens = torch.from_numpy(lens0.copy())
        kv.kv_splice_composed(st["desc"], st["bt"], st["max_blocks"], lens, s0, s1, nr,
                              stub_c, stub_r, ws)
        return kv.kv_last_launch_count()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    ms, kms, launches = _timed(call, K, W, prep=restore)
    seq_ms, _, _ = _timed(lambda: splice_step(st)[0], K, W, prep=restore)
    # end to end: directives are host arrays by design; the call plus a status read
    e2e_s = 0.0
    for _ in range(K):
        restore()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        call()
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        e2e_s += time.perf_counter() - t0
    barrier(world)
    clk = clocks.stop()
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    ms = max_over_ranks(ms, world)
    nbytes = rows * L * 2 * MLA_ROW_BYTES
    moved_successive = sum(rd["moved"] for rd in st["rounds"])
    peak, peak_kind = hbm_peak()
    achieved = nbytes / (kms * 1e-3) / 1e9
    out = {
        "metric": "relocated KV tokens/s (all layers)",
        "value": rows * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": f"leyline-splice-mla-composed: {L} layers, {S} sequences x "
                               f"{cfg['seq_len']} tokens, {R} directives per sequence (removing "
                               f"U[{cfg['span_lo']},{cfg['span_hi']}] tokens for a "
                               f"U[{cfg['stub_lo']},{cfg['stub_hi']}]-row stub each) as one "
                               "composed in-place edit",
                   "rows_moved_per_step_per_gpu": rows, "layers": L, "tiles": len(tiles),
                   "distinct_shifts": len(deltas),
                   "successive_calls_ms": seq_ms,
                   "successive_rows_moved": moved_successive,
                   "speedup_vs_successive": seq_ms / ms,
                   "parallelism": f"replicas x{world} (independent sequences)",
                   "l2": "inputs larger than L2 (%.1f GB moved per step); cache restored "
                         "from a pristine copy before each call, untimed" % (nbytes / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic("splice_mla_128k_composed"),
                     "kernel": "splice_composed_kernel<MLA>", "kernel_ms": kms,
                     "algorithmic_bytes_per_step": nbytes},
        "e2e": {"value": rows * world * K / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": int(len(tiles) * 48 + len(deltas) * 4),
                "d2h_bytes_per_step": 4},
        "clocks": clk, "gpu_launches": launches,
    }
    if args.check and rank == 0:
        import oracle as O
        restore()
        call()
        out["parity_sample"] = check_splice_sample(st, O.get(), composed=True)
    return out


# ---------------------------------------------------------------------------
# Workload: Kamera GQA relocation with a fused rank-16 patch
# ---------------------------------------------------------------------------

RELOC_GQA = dict(layers=32, num_reqs=16, chunks_per_req=64, chunk_len=576, delta_lo=0,
                 delta_hi=65536, n_pool_chunks=256, base_hi=32768, rank=16, std=0.02,
                 base=500000.0)
RELOC_GQA_SMALL = dict(RELOC_GQA, num_reqs=1, chunks_per_req=16, n_pool_chunks=16)


def build_relocate_gqa(rank: int, cfg, device: str = "cuda"):
    import position_independent_mla_gb300 as kv

    c = cfg
    wl = synth.relocate_workload(4004 + 100 * rank, num_reqs=c["num_reqs"],
                                 chunks_per_req=c["chunks_per_req"], len_lo=c["chunk_len"],
                                 len_hi=c["chunk_len"], delta_lo=c["delta_lo"],
                                 delta_hi=c["delta_hi"], n_pool_chunks=c["n_pool_chunks"],
                                 base_hi=c["base_hi"])
    L, W, m = c["layers"], 1024, c["rank"]
    src_k = torch.empty((L, wl.src_slots_total, W), dtype=torch.bfloat16, device=device)
    src_v = torch.empty((L, wl.src_slots_total, W), dtype=torch.bfloat16, device=device)
    fill_normal_(src_k, 4004 + 100 * rank)
    fill_normal_(src_v, 4005 + 100 * rank)
    dst_k = torch.zeros((L, wl.dst_slots_total, W), dtype=torch.bfloat16, device=device)
    dst_v = torch.zeros((L, wl.dst_slots_total, W), dtype=torch.bfloat16, device=device)
    sd = kv.pool_desc(src_v, src_k, 64, 8, c["base"])
    dd = kv.pool_desc(dst_v, dst_k, 64, 8, c["base"])
    g = torch.Generator(device=device)
    fac = {}
    for i, name in enumerate(("u_v", "u_k", "v_v", "v_k")):
        g.manual_seed(4100 + 100 * rank + i)
        shape = (L, wl.total_tokens, m) if name[0] == "u" else (L, wl.num_chunks, W, m)
        fac[name] = torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(c["std"])
    patch = kv.patch_desc(m, [fac["u_v"], fac["u_k"]], [fac["v_v"], fac["v_k"]])
    host = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).pin_memory()
            for k in ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta",
                      "block_tables")}
    dev = {k: v.to(device) for k, v in host.items()}
    ws = kv.workspace(dd, wl.total_tokens, wl.num_chunks, device=device)
    return dict(wl=wl, src_k=src_k, src_v=src_v, dst_k=dst_k, dst_v=dst_v, sd=sd, dd=dd,
                fac=fac, patch=patch, host=host, dev=dev, ws=ws, L=L, cfg=c)


def relocate_gqa_call(st, dev=None, stream=None, patch=True):
    import position_independent_mla_gb300 as kv

    wl, d = st["wl"], dev if dev is not None else st["dev"]
    kv.kv_relocate(st["sd"], st["dd"], wl.num_chunks, wl.total_tokens, d["tok_off"],
                   d["src_slots"], d["chunk_req"], d["chunk_dst_pos"], d["delta"],
                   d["block_tables"], wl.block_tables.shape[0], wl.block_tables.shape[1],
                   st["patch"] if patch else None, st["ws"], stream=stream)
    return kv.kv_last_launch_count()


def check_reloc_gqa_sample(st, orc, n_rows: int = 300, seed: int = 13) -> dict:
    """Sampled parity at full size: random (token, layer) rows, each checked
    against the oracle's fused relocation + patch on a one-token problem
    built from that row's source values and its U / V factors."""
    import oracle as O

    wl, L, m = st["wl"], st["L"], st["cfg"]["rank"]
    rng = np.random.default_rng(seed)
    worst = {"copy_beyond": 0, "rot_beyond": 0, "exact": 0, "one_ulp": 0, "values": 0}
    for _ in range(n_rows):
        t = int(rng.integers(wl.total_tokens))
        l = int(rng.integers(L))
        c = int(np.searchsorted(wl.tok_off, t, side="right") - 1)
        pos = int(wl.chunk_dst_pos[c]) + t - int(wl.tok_off[c])
        ds = int(wl.block_tables[wl.chunk_req[c], pos // 64]) * 64 + pos % 64
        ss = int(wl.src_slots[t])
        # a one-block pool holding the sampled source row in slot 0
        sv = np.zeros((1, 64, 1024), np.uint16)
        sk = np.zeros((1, 64, 1024), np.uint16)
        sv[0, 0] = synth.bits(st["src_v"][l, ss].cpu())
        sk[0, 0] = synth.bits(st["src_k"][l, ss].cpu())
        src = O.Pool(sv, sk, 64, 8, 128, st["cfg"]["base"])
        dst = O.Pool(np.zeros((1, 64, 1024), np.uint16), np.zeros((1, 64, 1024), np.uint16), 64, 8,
                     128, st["cfg"]["base"])
        u = [st["fac"][k][l, t].cpu().numpy().reshape(1, 1, m) for k in ("u_v", "u_k")]
        v = [st["fac"][k][l, c].cpu().numpy().reshape(1, 1, 1024, m) for k in ("v_v", "v_k")]
        assert orc.relocate(src, dst, [0, 1], [0], [0], [0], [int(wl.delta[c])], [[0]],
                            O.Patch(m, u, v)) == O.OK
        got_v = synth.bits(st["dst_v"][l, ds].cpu())
        got_k = synth.bits(st["dst_k"][l, ds].cpu())
        for got, want, key in ((got_v, dst.copy[0, 0], "copy_beyond"),
                               (got_k, dst.rot[0, 0], "rot_beyond")):
            r = ulp_stats(got, want)
            worst[key] += r["beyond"]
            worst["exact"] += r["exact"]
            worst["one_ulp"] += r["one_ulp"]
            worst["values"] += r["values"]
    worst["rows"] = n_rows
    return worst


def run_relocate_gqa_patch(args, rank, world, local):
    import position_independent_mla_gb300 as kv

    cfg = RELOC_GQA_SMALL if args.small else RELOC_GQA
    st = build_relocate_gqa(rank, cfg)
    wl, L, m = st["wl"], st["L"], cfg["rank"]
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        relocate_gqa_call(st)
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for a, b in ev:
        a.record()
        b.record()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    launches = 0
    t_start.record()
    for i in range(K):
        kv.kv_set_kernel_events(*ev[i])
        launches += relocate_gqa_call(st)
    t_stop.record()
    torch.cuda.synchronize()
    barrier(world)
    kv.kv_set_kernel_events(None, None)
    assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
    step_ms = t_start.elapsed_time(t_stop) / K
    kern_ms = sum(a.elapsed_time(b) for a, b in ev) / K

    # unfused comparison (relocation, then kv_patch on the relocated rows)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_unf = max(3, K // 4)
    e0.record()
    for _ in range(n_unf):
        relocate_gqa_call(st, patch=False)
        d = st["dev"]
        kv.kv_patch(st["dd"], wl.num_chunks, wl.total_tokens, d["tok_off"], d["chunk_req"],
                    d["chunk_dst_pos"], d["block_tables"], wl.block_tables.shape[0],
                    wl.block_tables.shape[1], st["patch"], st["ws"])
    e1.record()
    torch.cuda.synchronize()
    unfused_ms = e0.elapsed_time(e1) / n_unf
    # relocation alone (no patch): the plain GQA path
    e0.record()
    for _ in range(n_unf):
        relocate_gqa_call(st, patch=False)
    e1.record()
    torch.cuda.synchronize()
    reloc_only_ms = e0.elapsed_time(e1) / n_unf
    relocate_gqa_call(st)  # leave the fused result in place for the parity sample

    host, dev = st["host"], st["dev"]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(K):
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        relocate_gqa_call(st, dev)
        assert kv.kv_get_device_status(st["ws"], stream) == kv.KV_OK
    e2e_s = time.perf_counter() - t0
    clk = clocks.stop()
    step_ms = max_over_ranks(step_ms, world)
    e2e_s = max_over_ranks(e2e_s, world)

    T = wl.total_tokens
    kv_bytes = T * L * 2 * 2 * GQA_ROW_BYTES
    fac_bytes = T * L * 2 * m * 4 + wl.num_chunks * L * 2 * 1024 * m * 4
    bytes_per_launch = kv_bytes + fac_bytes + T * 4
    flops = T * L * 2 * 1024 * m * 2
    peak, peak_kind = hbm_peak()
    achieved = bytes_per_launch / (kern_ms * 1e-3) / 1e9
    out = {
        "metric": "relocated KV tokens/s (all layers)",
        "value": T * world / (step_ms * 1e-3), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": f"kamera-relocate-gqa-patch: {L} layers, K and V of 8 x 128 "
                               f"bf16, RoPE base 500000, {cfg['num_reqs']} requests x "
                               f"{cfg['chunks_per_req']} chunks of {cfg['chunk_len']} tokens, "
                               f"delta U[0,65536], fused rank-{m} fp32 patch on K and V",
                   "tokens_per_step_per_gpu": T, "layers": L, "chunks": wl.num_chunks,
                   "parallelism": f"replicas x{world} (independent batches)",
                   "l2": "inputs larger than L2 (%.1f GB moved per step)" % (bytes_per_launch / 1e9),
                   "unfused_relocate_then_patch_ms": unfused_ms,
                   "relocate_only_ms": reloc_only_ms,
                   "relocate_only_gbs": (wl.total_tokens * L * 2 * 2 * GQA_ROW_BYTES) /
                                        (reloc_only_ms * 1e-3) / 1e9},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic("relocate_gqa_patch"),
                     "kernel": "patch_tc_kernel (256-column slices, two heads)", "kernel_ms": kern_ms,
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "patch_tflops": flops / (kern_ms * 1e-3) / 1e12},
        "e2e": {"value": T * world * K / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "clocks": clk, "gpu_launches": launches,
    }
    if args.check and rank == 0:
        import oracle as O
        out["parity_sample"] = check_reloc_gqa_sample(st, O.get())
    return out


# ---------------------------------------------------------------------------
# Workload: one MLA layer, 4096 tokens, one directive (L2-resident)
# ---------------------------------------------------------------------------

SPLICE_4K = dict(layers=1, seq_len=4096, s_start=1024, s_end=2048, stub=16, base=10000.0)


def run_splice_mla_4k(args, rank, world, local):
    """Leyline splice of [1024, 2048) -> 16-row stub (Δ = -1008) on one MLA
    layer of 4096 tokens: 2048 downstream rows shifted and rotated.  The whole
    cache is 4.7 MB, so it lives in L2: reported warm, and cold with a 256 MB
    write before every step (outside the timed region).  A step is the whole
    kv_splice call (every operation it enqueues, timed with events around the
    call); the splice kernel alone is timed beside it."""
    import position_independent_mla_gb300 as kv

    c = SPLICE_4K
    ss = synth.splice_seqs(5005 + 100 * rank, [c["seq_len"]], c["seq_len"] // 64)
    pool = torch.empty((1, ss.num_slots, MLA_ROW), dtype=torch.bfloat16, device="cuda")
    fill_normal_(pool, 5005 + 100 * rank)
    pristine = pool.clone()
    stub_c = torch.empty((1, c["stub"], 512), dtype=torch.bfloat16, device="cuda")
    stub_r = torch.empty((1, c["stub"], 64), dtype=torch.bfloat16, device="cuda")
    fill_normal_(stub_c, 5006)
    fill_normal_(stub_r, 5007)
    desc = kv.pool_desc(pool[..., :512], pool[..., 512:], 64, 1, c["base"])
    bt = torch.from_numpy(ss.block_tables).cuda()
    ws = kv.workspace(desc, c["seq_len"], 1)
    s0, s1, nr = (torch.tensor([x], dtype=torch.int32) for x in (c["s_start"], c["s_end"], c["stub"]))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    moved = c["seq_len"] - c["s_end"] + c["stub"]

    def new_events(n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:   # torch creates the CUDA event on its first record()
            a.record()
            b.record()
        return evs

    def one(cold, call_ev, kern_ev):
        pool.copy_(pristine)
        if cold:
            flush.zero_()
        lens = torch.tensor([c["seq_len"]], dtype=torch.int32)
        kv.kv_set_kernel_events(*kern_ev)
        call_ev[0].record()
        kv.kv_splice(desc, 1, bt, ss.block_tables.shape[1], lens, s0, s1, nr, stub_c, stub_r,
                     kv.KV_AMORTIZE, ws)
        call_ev[1].record()
        kv.kv_set_kernel_events(None, None)
        return kv.kv_last_launch_count()

    res, kres = {}, {}
    launches = 0
    clocks = ClockSampler(local)
    clocks.start()
    for cold in (False, True):
        for _ in range(args.warmup):
            one(cold, *new_events(2))
        calls, kerns = new_events(args.steps), new_events(args.steps)
        torch.cuda.synchronize()
        for ce, ke in zip(calls, kerns):
            launches += one(cold, ce, ke)
        torch.cuda.synchronize()
        key = "cold" if cold else "warm"
        res[key] = sum(a.elapsed_time(b) for a, b in calls) / args.steps
        kres[key] = sum(a.elapsed_time(b) for a, b in kerns) / args.steps
    # end to end through the C ABI: per step the stub rows come from pinned
    # host memory, then the call and a status read-back (cache restored and
    # L2 flushed before each step, untimed)
    hc, hr = stub_c.cpu().pin_memory(), stub_r.cpu().pin_memory()
    e2e_s = 0.0
    for _ in range(args.steps):
        pool.copy_(pristine)
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        stub_c.copy_(hc, non_blocking=True)
        stub_r.copy_(hr, non_blocking=True)
        lens = torch.tensor([c["seq_len"]], dtype=torch.int32)
        kv.kv_splice(desc, 1, bt, ss.block_tables.shape[1], lens, s0, s1, nr, stub_c, stub_r,
                     kv.KV_AMORTIZE, ws)
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        e2e_s += time.perf_counter() - t0
    clk = clocks.stop()
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    bytes_step = moved * 2 * MLA_ROW_BYTES
    peak, peak_kind = hbm_peak()
    ms, kms = res["cold"], kres["cold"]
    out = {
        "metric": "relocated KV tokens/s (all layers)", "value": moved * world / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": "leyline-splice-mla-4k: 1 layer, 4096 tokens, [1024,2048) -> "
                               "16-row stub (delta -1008), 2048 rows shifted",
                   "l2": "cache of 4.7 MB is L2-resident; value is cold (256 MB written "
                         "before each step, untimed); warm given beside it",
                   "warm_ms": res["warm"], "cold_ms": res["cold"],
                   "warm_kernel_ms": kres["warm"], "cold_kernel_ms": kres["cold"],
                   "warm_tokens_per_s": moved / (res["warm"] * 1e-3),
                   "step": "the whole kv_splice call (events around it)"},
        "roofline": {"bound": "hbm", "achieved": bytes_step / (kms * 1e-3) / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": bytes_step / (kms * 1e-3) / 1e9 / peak,
                     "peak_kind": peak_kind, "traffic": None, "kernel": "splice_kernel<MLA>",
                     "kernel_ms": kms, "algorithmic_bytes_per_launch": bytes_step,
                     "note": "4.7 MB edit: one wave of 65 blocks, bound by launch and "
                             "per-block latency, not by HBM bandwidth; the fraction is "
                             "reported against the HBM copy peak for form"},
        "e2e": {"value": moved * world * args.steps / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": int(hc.numel() * 2 + hr.numel() * 2),
                "d2h_bytes_per_step": 4,
                "copies": "the stub rows from pinned host memory; the directive goes by value "
                          "in the launch"},
        "clocks": clk, "gpu_launches": launches,
    }
    return out


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    import oracle as O

    if rank != 0:
        return None
    orc = O.get()
    c = RELOC_MLA
    # calibrate, then size each step so the whole run stays within ~2 minutes
    probe_tokens = 32

    def step(n_tok, seed):
        wl = synth.relocate_workload(seed, num_reqs=1, chunks_per_req=1, len_lo=n_tok,
                                     len_hi=n_tok, delta_lo=c["delta_lo"], delta_hi=c["delta_hi"],
                                     n_pool_chunks=1, base_hi=63)
        L = c["layers"]
        src = O.Pool(synth.bits(synth.bf16_normal((L, wl.src_slots_total, 512), seed)).copy(),
                     synth.bits(synth.bf16_normal((L, wl.src_slots_total, 64), seed + 1)).copy(),
                     64, 1, 64, c["base"])
        dst = O.Pool(np.zeros((L, wl.dst_slots_total, 512), np.uint16),
                     np.zeros((L, wl.dst_slots_total, 64), np.uint16), 64, 1, 64, c["base"])
        t0 = time.perf_counter()
        assert orc.relocate(src, dst, wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos,
                            wl.delta, wl.block_tables) == O.OK
        return time.perf_counter() - t0

    rate = probe_tokens / step(probe_tokens, 5)
    per_core = int(max(16, min(4096, rate * 120.0 / max(1, args.steps + args.warmup))))
    cores = OracleCores()  # one process per host core, spawned before any timing
    try:
        cores.run("relocate-mla", 16, 1)
        for w in range(args.warmup):
            cores.run("relocate-mla", per_core, 10 + w)
        total, ntok = 0.0, 0
        for k in range(args.steps):
            n, dt, _ = cores.run("relocate-mla", per_core, 1000 + 131 * k)
            ntok += n
            total += dt
    finally:
        cores.close()
    value = ntok / total
    per_step = per_core * cores.n
    return {
        "metric": "relocated KV tokens/s (all layers)", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": "irminsul-relocate-mla (bounded sample per step: "
                               f"{cores.n} independent chunks of {per_core} tokens, one per "
                               "host core, 61 layers)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores.n, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"{per_step} tokens x 61 layers per step, "
                                   f"{per_core} per core"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# Workload: Kamera sliding window (GQA): survival by remapping + recall
# ---------------------------------------------------------------------------

WINDOW_GQA = dict(layers=32, num_reqs=16, window=64, chunk_len=576, slide=8, n_canon=256,
                  rank=16, std=0.02, base=500000.0)
# A small case of the same kernels (~1.3 GB).
WINDOW_GQA_SMALL = dict(WINDOW_GQA, num_reqs=1, window=16, slide=4, n_canon=32)


def build_window_gqa(rank: int, cfg):
    """A canonical store (chunks prefilled alone at position 0, GQA K and V,
    one rank-m patch per canonical chunk and channel) and a per-request
    window of `window` chunks filled from it."""
    import position_independent_mla_gb300 as kv

    c = cfg
    L, R, W, cl, m, W1 = c["layers"], c["num_reqs"], c["window"], c["chunk_len"], c["rank"], 1024
    nc = c["n_canon"]
    reg_k = torch.empty((L, nc * cl, W1), dtype=torch.bfloat16, device="cuda")
    reg_v = torch.empty_like(reg_k)
    fill_normal_(reg_k, 7007 + 100 * rank)
    fill_normal_(reg_v, 7008 + 100 * rank)
    g = torch.Generator(device="cuda")
    g.manual_seed(7009 + 100 * rank)
    u = [torch.randn((L, nc * cl, m), generator=g, device="cuda").mul_(c["std"]) for _ in range(2)]
    v = [torch.randn((L, nc, W1, m), generator=g, device="cuda").mul_(c["std"]) for _ in range(2)]
    mb = W * cl // 64
    win_k = torch.zeros((L, R * mb * 64, W1), dtype=torch.bfloat16, device="cuda")
    win_v = torch.zeros_like(win_k)
    rng = np.random.default_rng(7010 + 100 * rank)
    bt0 = rng.permutation(R * mb).astype(np.int32).reshape(R, mb)
    ids = np.array([[(r * W + j) % nc for j in range(W)] for r in range(R)], np.int64)
    st = dict(cfg=c, L=L, R=R, W=W, cl=cl, m=m, mb=mb, ids=ids, bt0=bt0, u=u, v=v,
              reg_k=reg_k, reg_v=reg_v, win_k=win_k, win_v=win_v,
              sd=kv.pool_desc(reg_v, reg_k, 64, 8, c["base"]),
              wd=kv.pool_desc(win_v, win_k, 64, 8, c["base"]),
              bt=torch.from_numpy(bt0.copy()).cuda())
    st["ws"] = kv.workspace(st["wd"], R * W * cl, R * W)
    return st


def window_recall_args(st, chunks, slot0):
    """kv_relocate arguments bringing canonical chunks[r][j] of each request r
    to window positions (slot0 + j) * chunk_len, with their stored patches."""
    import position_independent_mla_gb300 as kv

    R, cl = st["R"], st["cl"]
    n = chunks.shape[1]
    ids = chunks.reshape(-1)
    pos = np.tile((slot0 + np.arange(n)) * cl, R).astype(np.int32)
    args = dict(
        tok_off=(np.arange(R * n + 1) * cl).astype(np.int32),
        src_slots=(ids[:, None] * cl + np.arange(cl)[None, :]).reshape(-1).astype(np.int32),
        chunk_req=np.repeat(np.arange(R), n).astype(np.int32), chunk_dst_pos=pos,
        delta=pos.copy())                                  # canonical chunks sit at position 0
    dev = {k: torch.from_numpy(v_).cuda() for k, v_ in args.items()}
    pd = kv.patch_desc(st["m"], st["u"], st["v"], torch.from_numpy(ids * cl).cuda(),
                       torch.from_numpy(ids.astype(np.int32)).cuda())
    return dict(host=args, dev=dev, pd=pd, n=R * n)


def window_relocate(st, ra):
    import position_independent_mla_gb300 as kv

    d, cl = ra["dev"], st["cl"]
    kv.kv_relocate(st["sd"], st["wd"], ra["n"], ra["n"] * cl, d["tok_off"], d["src_slots"],
                   d["chunk_req"], d["chunk_dst_pos"], d["delta"], st["bt"], st["R"], st["mb"],
                   ra["pd"], st["ws"])
    return kv.kv_last_launch_count()


def window_slide(st, mode):
    import position_independent_mla_gb300 as kv

    R, W, cl, sl = st["R"], st["W"], st["cl"], st["cfg"]["slide"]
    lens = torch.full((R,), W * cl, dtype=torch.int32)
    z = torch.zeros(R, dtype=torch.int32)
    kv.kv_splice(st["wd"], R, st["bt"], st["mb"], lens, z, torch.full((R,), sl * cl,
                 dtype=torch.int32), z, None, None, mode, st["ws"])
    return kv.kv_last_launch_count()


def check_window_sample(st, recall, orc, n_rows: int = 120, seed: int = 17) -> dict:
    """After one step from a fresh window: survivors are their first placement
    turned by R(-slide * chunk_len) (rotary part) and unchanged otherwise;
    recalled chunks are a fresh relocation + stored patch at the window's end.
    Each sampled row is rebuilt by the oracle on a one-token problem."""
    import oracle as O

    c, L, cl, W, sl = st["cfg"], st["L"], st["cl"], st["W"], st["cfg"]["slide"]
    rng = np.random.default_rng(seed)
    bt = st["bt"].cpu().numpy()
    out = {"v_beyond": 0, "k_beyond": 0, "exact": 0, "one_ulp": 0, "values": 0}
    for _ in range(n_rows):
        r, p, l = int(rng.integers(st["R"])), int(rng.integers(W * cl)), int(rng.integers(L))
        j, i = p // cl, p % cl
        survivor = j < W - sl
        cid = int(st["ids"][r, j + sl] if survivor else st["ids"][r, j - (W - sl)])
        p0 = p + sl * cl if survivor else p               # position of its relocation
        row = cid * cl + i
        sv = np.zeros((1, 64, 1024), np.uint16)
        sk = np.zeros((1, 64, 1024), np.uint16)
        sv[0, 0] = synth.bits(st["reg_v"][l, row].cpu())
        sk[0, 0] = synth.bits(st["reg_k"][l, row].cpu())
        src = O.Pool(sv, sk, 64, 8, 128, c["base"])
        dst = O.Pool(np.zeros_like(sv), np.zeros_like(sk), 64, 8, 128, c["base"])
        u = [x[l, row].cpu().numpy().reshape(1, 1, -1) for x in st["u"]]
        v = [x[l, cid].cpu().numpy().reshape(1, 1, 1024, -1) for x in st["v"]]
        # canonical chunks were prefilled from position 0: δ is the chunk's start
        assert orc.relocate(src, dst, [0, 1], [0], [0], [0], [p0 - i], [[0]],
                            O.Patch(st["m"], u, v)) == O.OK
        want_v, want_k = dst.copy[0, 0], dst.rot[0, 0]
        if survivor:
            want_k = np.concatenate([orc.rotate_bf16(want_k[h * 128:(h + 1) * 128], -sl * cl,
                                                     c["base"]) for h in range(8)])
        slot = int(bt[r, p // 64]) * 64 + p % 64
        got_v = synth.bits(st["win_v"][l, slot].cpu())
        got_k = synth.bits(st["win_k"][l, slot].cpu())
        for got, want, key in ((got_v, want_v, "v_beyond"), (got_k, want_k, "k_beyond")):
            rs = ulp_stats(got, want)
            out[key] += rs["beyond"]
            out["exact"] += rs["exact"]
            out["one_ulp"] += rs["one_ulp"]
            out["values"] += rs["values"]
    out["rows"] = n_rows
    return out


def run_window_gqa(args, rank, world, local):
    """Kamera's sliding window, GQA, in steady state: each step evicts the
    `slide` oldest chunks of every request's window (survival: the survivors'
    K turned by R(-slide * chunk_len), no patch, by block-table remapping) and
    recalls them at the window's end from the canonical store with their
    stored rank-16 patches (relocation + patch through the factor maps), so
    the window cycles.  Timed against the same step with a data-moving slide."""
    import position_independent_mla_gb300 as kv

    cfg = WINDOW_GQA_SMALL if args.small else WINDOW_GQA
    st = build_window_gqa(rank, cfg)
    L, R, W, cl, sl, m = st["L"], st["R"], st["W"], st["cl"], cfg["slide"], st["m"]
    window_relocate(st, window_recall_args(st, st["ids"], 0))      # fill, untimed
    phases = W // sl
    recalls = [window_recall_args(st, np.roll(st["ids"], -k * sl, axis=1)[:, W - sl:], W - sl)
               for k in range(1, phases + 1)]
    out_check = None
    if args.check and rank == 0:
        import oracle as O
        window_slide(st, kv.KV_AMORTIZE_REMAP)
        window_relocate(st, recalls[0])
        out_check = check_window_sample(st, recalls[0], O.get())
        st["bt"].copy_(torch.from_numpy(st["bt0"]))                # start over
        window_relocate(st, window_recall_args(st, st["ids"], 0))
    step_no = [0]

    def step(mode):
        def call():
            n = window_slide(st, mode)
            n += window_relocate(st, recalls[step_no[0] % phases])
            step_no[0] += 1
            return n
        return call

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    K, Wu = args.steps, args.warmup
    ms, _, launches = _timed(step(kv.KV_AMORTIZE_REMAP), K, Wu)
    amortize_ms, _, _ = _timed(step(kv.KV_AMORTIZE), K, Wu)
    # the two halves of a step, each between events on the stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for k in range(K):
        ev[k][0].record()
        window_slide(st, kv.KV_AMORTIZE_REMAP)
        ev[k][1].record()
        window_relocate(st, recalls[step_no[0] % phases])
        step_no[0] += 1
        ev[k][2].record()
    torch.cuda.synchronize()
    slide_ms = float(np.median([e[0].elapsed_time(e[1]) for e in ev]))
    recall_ms = float(np.median([e[1].elapsed_time(e[2]) for e in ev]))
    barrier(world)
    clk = clocks.stop()
    assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
    ms = max_over_ranks(ms, world)
    surv, rec = R * (W - sl) * cl, R * sl * cl
    nbytes = (surv * L * 2 * 2048 + rec * (L * (2 * 4096 + 2 * m * 4) + 4) +
              R * sl * L * 2 * 1024 * m * 4)
    peak, peak_kind = hbm_peak()
    out = {
        "metric": "relocated KV tokens/s (all layers)",
        "value": (surv + rec) * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": Wu, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "impl": "ours",
        "config": {"workload": f"kamera-window-gqa: {L} layers, K and V of 8 x 128, {R} "
                               f"requests x a window of {W} chunks of {cl} tokens; each step "
                               f"evicts the {sl} oldest chunks (survivors re-rotated by block-"
                               f"table remapping) and recalls them at the end from the canonical "
                               f"store with their stored rank-{m} patches",
                   "survivor_rows": surv, "recalled_rows": rec, "layers": L,
                   "amortize_slide_ms": amortize_ms, "speedup_vs_amortize": amortize_ms / ms,
                   "slide_ms": slide_ms, "recall_ms": recall_ms,
                   "slide_gbs": surv * L * 2 * 2048 / (slide_ms * 1e-3) / 1e9,
                   "parallelism": f"replicas x{world} (independent requests)",
                   "l2": "inputs larger than L2 (%.1f GB moved per step)" % (nbytes / 1e9)},
        "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": nbytes / (ms * 1e-3) / 1e9 / peak,
                     "peak_kind": peak_kind, "traffic": recorded_traffic("window_gqa"),
                     "kernel": "remap_data_kernel<GQA> + patch_tc_kernel (whole step)",
                     "algorithmic_bytes_per_step": nbytes},
        "e2e": None, "clocks": clk, "gpu_launches": launches,
    }
    if out_check is not None:
        out["parity_sample"] = out_check
    return out


# ---------------------------------------------------------------------------
# Workload: MLA sweep over chunk length x δ (relocate; splice with Δ = δ; patch)
# ---------------------------------------------------------------------------

SWEEP_MLA = dict(layers=61, chunk_lens=(16, 64, 256, 1024, 4096),
                 deltas=(1, -1, 1000, -1000, 100000, -100000), num_reqs=8, req_tokens=131072,
                 rank=8, base=10000.0, splice_seq=131072)
# A small case of the same kernels for counter captures: 16 layers x 4 x 16,384
# tokens, 2.4 GB moved per relocation call (19x the L2), a few GB on the device.
SWEEP_MLA_SMALL = dict(SWEEP_MLA, layers=16, num_reqs=4, req_tokens=16384,
                       deltas=(1, -1, 1000, -1000, 10000, -10000), splice_seq=16384)


def _timed(call, K: int, W: int, prep=None):
    """W untimed calls, then K timed ones, each after `prep` (untimed).
    Returns (median call ms, median kernel ms, kernels launched while timed);
    the kernel time is the library's own event pair around its main kernel."""
    import position_independent_mla_gb300 as kv

    for _ in range(W):
        if prep:
            prep()
        call()
    torch.cuda.synchronize()
    call_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    kern_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    for a, b in call_ev + kern_ev:
        a.record()
        b.record()
    launches = 0
    for i in range(K):
        if prep:
            prep()
        call_ev[i][0].record()
        kv.kv_set_kernel_events(*kern_ev[i])
        launches += call()
        call_ev[i][1].record()
    torch.cuda.synchronize()
    kv.kv_set_kernel_events(None, None)
    call_ms = float(np.median([a.elapsed_time(b) for a, b in call_ev]))
    kern_ms = float(np.median([a.elapsed_time(b) for a, b in kern_ev]))
    return call_ms, kern_ms, launches


def check_patch_sample(rows_before, rows_after, idx, wl, u, v, m, orc) -> dict:
    """Sampled parity of the standalone patch: each sampled (token, layer) row,
    as stored before the call, patched by the oracle on a one-token problem."""
    import oracle as O

    out = {"copy_beyond": 0, "rot_beyond": 0, "exact": 0, "one_ulp": 0, "values": 0}
    for k, (t, l) in enumerate(idx):
        c = int(np.searchsorted(wl.tok_off, t, side="right") - 1)
        pc, pr = np.zeros((1, 64, 512), np.uint16), np.zeros((1, 64, 64), np.uint16)
        pc[0, 0], pr[0, 0] = rows_before[k, :512], rows_before[k, 512:]
        pool = O.Pool(pc, pr, 64, 1, 64, 10000.0)
        ut = u[l, t].cpu().numpy().reshape(1, 1, m)
        vc = v[l, c].cpu().numpy().reshape(1, 1, 576, m)
        assert orc.patch_apply(pool, [0, 1], [0], [0], [[0]],
                               O.Patch(m, [ut, ut], [vc[:, :, :512], vc[:, :, 512:]])) == O.OK
        for g, want, key in ((rows_after[k, :512], pool.copy[0, 0], "copy_beyond"),
                             (rows_after[k, 512:], pool.rot[0, 0], "rot_beyond")):
            r = ulp_stats(g, want)
            out[key] += r["beyond"]
            out["exact"] += r["exact"]
            out["one_ulp"] += r["one_ulp"]
            out["values"] += r["values"]
    out["rows"] = len(idx)
    return out


def run_sweep_mla(args, rank, world, local):
    """MLA, 61 layers: relocation at every (chunk length, δ) point; the
    standalone rank-8 patch per chunk length; the splice with Δ = δ per δ (on
    one sequence). Each measurement is the median of `--steps` calls."""
    import position_independent_mla_gb300 as kv

    cfg = SWEEP_MLA_SMALL if args.small else SWEEP_MLA
    L, R, N, m, base = cfg["layers"], cfg["num_reqs"], cfg["req_tokens"], cfg["rank"], cfg["base"]
    K, W = args.steps, args.warmup
    peak, peak_kind = hbm_peak()
    orc = None
    if args.check and rank == 0:
        import oracle as O
        orc = O.get()
    clocks = ClockSampler(local)
    clocks.start()
    launches = 0

    # --- relocation: one registry of R*N distinct rows, one destination pool
    wl0 = synth.fixed_chunk_workload(0, cfg["chunk_lens"][0], 0, R, N)
    src = torch.empty((L, wl0.src_slots_total, MLA_ROW), dtype=torch.bfloat16, device="cuda")
    fill_normal_(src, 5005 + 100 * rank)
    dst = torch.zeros((L, wl0.dst_slots_total, MLA_ROW), dtype=torch.bfloat16, device="cuda")
    sd = kv.pool_desc(src[..., :512], src[..., 512:], 64, 1, base)
    dd = kv.pool_desc(dst[..., :512], dst[..., 512:], 64, 1, base)
    reloc, wls = [], {}
    for i, cl in enumerate(cfg["chunk_lens"]):
        for j, delta in enumerate(cfg["deltas"]):
            wl = synth.fixed_chunk_workload(5100 + 100 * rank + 10 * i + j, cl, delta, R, N)
            wls.setdefault(cl, wl)
            host = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).pin_memory()
                    for k in ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta",
                              "block_tables")}
            d = {k: v.cuda() for k, v in host.items()}
            ws = kv.workspace(dd, wl.total_tokens, wl.num_chunks)

            def call(wl=wl, d=d, ws=ws):
                kv.kv_relocate(sd, dd, wl.num_chunks, wl.total_tokens, d["tok_off"],
                               d["src_slots"], d["chunk_req"], d["chunk_dst_pos"], d["delta"],
                               d["block_tables"], R, wl.block_tables.shape[1], None, ws)
                return kv.kv_last_launch_count()

            ms, kms, n = _timed(call, K, W)
            launches += n
            assert kv.kv_get_device_status(ws) == kv.KV_OK
            # end to end: the index arrays from pinned host memory, the call, a
            # status read-back
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(K):
                for k2 in host:
                    d[k2].copy_(host[k2], non_blocking=True)
                call()
                assert kv.kv_get_device_status(ws) == kv.KV_OK
            e2e_ms = (time.perf_counter() - t0) / K * 1e3
            T = wl.total_tokens
            nbytes = T * (L * 2 * MLA_ROW_BYTES + 4)
            pt = {"chunk_len": cl, "delta": delta, "chunks": wl.num_chunks, "ms": ms,
                  "kernel_ms": kms, "tokens_per_s": T / (ms * 1e-3),
                  "gbs": nbytes / (kms * 1e-3) / 1e9, "frac": nbytes / (kms * 1e-3) / 1e9 / peak,
                  "bytes": nbytes, "e2e_ms": e2e_ms,
                  "h2d_bytes": sum(t.numel() * t.element_size() for t in host.values())}
            if orc is not None:
                pt["parity_sample"] = check_relocate_sample(
                    dict(wl=wl, L=L, src=src, dst=dst, cfg=cfg), orc, n_rows=300, seed=7 + j)
            reloc.append(pt)
    del src
    torch.cuda.empty_cache()

    # --- standalone patch (in place on the relocated destination), per chunk length
    patch = []
    for i, cl in enumerate(cfg["chunk_lens"]):
        wl = wls[cl]
        T, C = wl.total_tokens, wl.num_chunks
        g = torch.Generator(device="cuda")
        g.manual_seed(5600 + 100 * rank + i)
        u = torch.randn((L, T, m), generator=g, device="cuda").mul_(0.02)
        v = torch.randn((L, C, 576, m), generator=g, device="cuda").mul_(0.02)
        pd = kv.patch_desc(m, [u, u], [v[:, :, :512], v[:, :, 512:]])
        d = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).cuda()
             for k in ("tok_off", "chunk_req", "chunk_dst_pos", "block_tables")}
        ws = kv.workspace(dd, T, C)

        def call(wl=wl, d=d, ws=ws, pd=pd):
            kv.kv_patch(dd, wl.num_chunks, wl.total_tokens, d["tok_off"], d["chunk_req"],
                        d["chunk_dst_pos"], d["block_tables"], R, wl.block_tables.shape[1], pd, ws)
            return kv.kv_last_launch_count()

        pt = {"chunk_len": cl, "chunks": C}
        if orc is not None:
            rng = np.random.default_rng(31 + i)
            idx = [(int(rng.integers(T)), int(rng.integers(L))) for _ in range(100)]

            def rows(idx=idx, wl=wl):
                out = []
                for t, l in idx:
                    c = int(np.searchsorted(wl.tok_off, t, side="right") - 1)
                    p = int(wl.chunk_dst_pos[c]) + t - int(wl.tok_off[c])
                    slot = int(wl.block_tables[wl.chunk_req[c], p // 64]) * 64 + p % 64
                    out.append(synth.bits(dst[l, slot].cpu()))
                return np.stack(out)

            before = rows()
            call()
            pt["parity_sample"] = check_patch_sample(before, rows(), idx, wl, u, v, m, orc)
        ms, kms, n = _timed(call, K, W)
        launches += n
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        nbytes = T * L * 2 * MLA_ROW_BYTES + T * L * m * 4 + C * L * 576 * m * 4
        pt.update({"ms": ms, "kernel_ms": kms, "tokens_per_s": T / (ms * 1e-3),
                   "gbs": nbytes / (kms * 1e-3) / 1e9,
                   "frac": nbytes / (kms * 1e-3) / 1e9 / peak, "bytes": nbytes})
        patch.append(pt)
        del u, v, pd
    del dst
    torch.cuda.empty_cache()

    # --- splice with Δ = δ on one sequence: n_R = max(16, 16 + δ), |S| = n_R - δ
    n = cfg["splice_seq"]
    max_blocks = (n + max(cfg["deltas"]) + 63) // 64
    ss = synth.splice_seqs(5700 + 100 * rank, [n], max_blocks)
    pool = torch.empty((L, ss.num_slots, MLA_ROW), dtype=torch.bfloat16, device="cuda")
    fill_normal_(pool, 5701 + 100 * rank)
    pristine = pool.clone()
    desc = kv.pool_desc(pool[..., :512], pool[..., 512:], 64, 1, base)
    bt = torch.from_numpy(ss.block_tables).cuda()
    ws = kv.workspace(desc, n, 1)
    splice = []
    for j, delta in enumerate(cfg["deltas"]):
        nr = max(16, 16 + delta)
        span = nr - delta
        rng = np.random.default_rng(5800 + 100 * rank + j)
        s0 = int(rng.integers(0, n - span + 1))
        d = synth.Directives(np.asarray([s0], np.int32), np.asarray([s0 + span], np.int32),
                             np.asarray([nr], np.int32))
        stub_c = torch.empty((L, nr, 512), dtype=torch.bfloat16, device="cuda")
        stub_r = torch.empty((L, nr, 64), dtype=torch.bfloat16, device="cuda")
        fill_normal_(stub_c, 5900 + 100 * rank + j)
        fill_normal_(stub_r, 5950 + 100 * rank + j)
        args_h = [torch.from_numpy(x.copy()) for x in (d.s_start, d.s_end, d.stub_len)]

        def call(args_h=args_h, stub_c=stub_c, stub_r=stub_r):
            lens = torch.tensor([n], dtype=torch.int32)
            kv.kv_splice(desc, 1, bt, max_blocks, lens, *args_h, stub_c, stub_r,
                         kv.KV_AMORTIZE, ws)
            return kv.kv_last_launch_count()

        ms, kms, k_l = _timed(call, K, W, prep=lambda: pool.copy_(pristine))
        launches += k_l
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        moved = (n - (s0 + span)) + nr
        nbytes = moved * L * 2 * MLA_ROW_BYTES
        pt = {"delta": delta, "stub_rows": nr, "removed": span, "s_start": s0,
              "rows_moved": moved, "ms": ms, "kernel_ms": kms,
              "tokens_per_s": moved / (ms * 1e-3), "gbs": nbytes / (kms * 1e-3) / 1e9,
              "frac": nbytes / (kms * 1e-3) / 1e9 / peak, "bytes": nbytes,
              "l2": "larger than L2" if nbytes > 2 * 129e6 else "L2-resident"}
        if orc is not None:
            pool.copy_(pristine)
            call()
            pt["parity_sample"] = check_splice_sample(
                dict(L=L, S=1, ss=ss, cfg=cfg, rounds=[dict(d=d, stub_c=stub_c, stub_r=stub_r)],
                     final_lens=np.asarray([n + delta]), pristine=pristine, pool=pool),
                orc, n_rows=300, seed=13 + j)
        splice.append(pt)
        del stub_c, stub_r
    clk = clocks.stop()

    tot_tok = sum(p["chunks"] * p["chunk_len"] for p in reloc)
    tot_ms = sum(p["ms"] for p in reloc)
    tot_bytes = sum(p["bytes"] for p in reloc)
    tot_kms = sum(p["kernel_ms"] for p in reloc)
    tot_e2e_ms = sum(p["e2e_ms"] for p in reloc)
    achieved = tot_bytes / (tot_kms * 1e-3) / 1e9
    return {
        "metric": "relocated KV tokens/s (all layers)",
        "value": tot_tok * world / (tot_ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": tot_ms / len(reloc), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "impl": "ours",
        "config": {"workload": f"mla-sweep: {L} layers, {R} requests x {N} tokens per "
                               "relocation, chunk lengths x delta; splice with Delta = delta "
                               f"on one {n}-token sequence; standalone rank-{m} patch",
                   "value_is": "relocated tokens over all points / relocation time over all points",
                   "steps_per_point": K, "warmup_per_point": W,
                   "relocate_frac_min_max": [min(p["frac"] for p in reloc),
                                             max(p["frac"] for p in reloc)],
                   "splice_frac_by_delta": {str(p["delta"]): round(p["frac"], 3) for p in splice},
                   "patch_frac_by_chunk_len": {str(p["chunk_len"]): round(p["frac"], 3)
                                               for p in patch},
                   "relocate": reloc, "splice": splice, "patch": patch,
                   "l2": "relocation and patch move >= 4 GB per call; splice points say"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic("sweep_mla"),
                     "kernel": "relocate_kernel<MLA> over all sweep points",
                     "kernel_ms": tot_kms / len(reloc),
                     "algorithmic_bytes_per_launch": tot_bytes / len(reloc)},
        "e2e": {"value": tot_tok * world / (tot_e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": sum(p["h2d_bytes"] for p in reloc) / len(reloc),
                "d2h_bytes_per_step": 4,
                "copies": "per relocation call: its index arrays from pinned host memory and "
                          "the status word back"},
        "clocks": clk, "gpu_launches": launches,
    }


# ---------------------------------------------------------------------------
# Workload: the other row families (GQA 4 x 128, MHA 32 x 128) and
# interleaved RoPE pairs (MLA), relocation without a patch
# ---------------------------------------------------------------------------

FAMILIES = [
    # name, layers, copy_dim, rot heads, head dim, rope base, pairs, requests, chunks/req, chunk len
    dict(name="gqa4-qwen2.5-7b", layers=28, copy_dim=512, heads=4, hd=128, base=1000000.0,
         il=0, num_reqs=16, chunks_per_req=64, chunk_len=576, n_pool_chunks=256),
    dict(name="mha-llama2-7b", layers=32, copy_dim=4096, heads=32, hd=128, base=10000.0,
         il=0, num_reqs=8, chunks_per_req=32, chunk_len=512, n_pool_chunks=128),
    dict(name="mla-interleaved", layers=61, copy_dim=512, heads=1, hd=64, base=10000.0,
         il=1, num_reqs=32, chunks_per_req=16, chunk_len=1152, n_pool_chunks=256),
]


def check_family_sample(fam, wl, src_c, src_r, dst_c, dst_r, orc, n_rows=200, seed=19) -> dict:
    """Sampled parity: random (token, layer) rows of the relocation; copy part
    against the source row, every rotary head against the oracle's rotation."""
    rng = np.random.default_rng(seed)
    toks = rng.integers(0, wl.total_tokens, n_rows)
    lays = rng.integers(0, fam["layers"], n_rows)
    chunk = np.searchsorted(wl.tok_off, toks, side="right") - 1
    pos = wl.chunk_dst_pos[chunk] + (toks - wl.tok_off[chunk])
    dslot = wl.block_tables[wl.chunk_req[chunk], pos // 64].astype(np.int64) * 64 + pos % 64
    sslot = wl.src_slots[toks].astype(np.int64)
    li = torch.from_numpy(lays).cuda()
    s_c = synth.bits(src_c[li, torch.from_numpy(sslot).cuda()].cpu())
    d_c = synth.bits(dst_c[li, torch.from_numpy(dslot).cuda()].cpu())
    s_r = synth.bits(src_r[li, torch.from_numpy(sslot).cuda()].cpu())
    d_r = synth.bits(dst_r[li, torch.from_numpy(dslot).cuda()].cpu())
    hd = fam["hd"]
    want = np.stack([np.concatenate([orc.rotate_bf16(s_r[i, h * hd:(h + 1) * hd],
                                                     int(wl.delta[chunk[i]]), fam["base"],
                                                     interleaved=bool(fam["il"]))
                                     for h in range(fam["heads"])]) for i in range(n_rows)])
    r = ulp_stats(d_r, want)
    return {"rows": n_rows, "copy_rows_differing": int((s_c != d_c).any(axis=1).sum()),
            "rot_exact": r["exact"], "rot_one_ulp": r["one_ulp"], "rot_beyond": r["beyond"]}


def run_families(args, rank, world, local):
    """Relocation (no patch) for the row families beside the headline MLA: GQA with
    4 KV heads (Qwen2.5-7B shape), MHA with 32 heads (Llama-2-7B shape), and MLA
    rows whose k_pe pairs are interleaved -- one line, one entry per family."""
    import position_independent_mla_gb300 as kv

    K, W = args.steps, args.warmup
    peak, peak_kind = hbm_peak()
    clocks = ClockSampler(local)
    clocks.start()
    res, tot_tok, tot_ms, launches, main = [], 0, 0.0, 0, None
    orc = None
    if args.check and rank == 0:
        import oracle as O
        orc = O.get()
    for fam in FAMILIES:
        f = dict(fam)
        if args.small:
            f.update(num_reqs=1, n_pool_chunks=16)
        wl = synth.relocate_workload(6006 + 100 * rank, num_reqs=f["num_reqs"],
                                     chunks_per_req=f["chunks_per_req"], len_lo=f["chunk_len"],
                                     len_hi=f["chunk_len"], delta_lo=-32768, delta_hi=32768,
                                     n_pool_chunks=f["n_pool_chunks"], base_hi=32768)
        L, rw = f["layers"], f["heads"] * f["hd"]
        src_c = torch.empty((L, wl.src_slots_total, f["copy_dim"]), dtype=torch.bfloat16,
                            device="cuda")
        src_r = torch.empty((L, wl.src_slots_total, rw), dtype=torch.bfloat16, device="cuda")
        fill_normal_(src_c, 6007)
        fill_normal_(src_r, 6008)
        dst_c = torch.zeros((L, wl.dst_slots_total, f["copy_dim"]), dtype=torch.bfloat16,
                            device="cuda")
        dst_r = torch.zeros((L, wl.dst_slots_total, rw), dtype=torch.bfloat16, device="cuda")
        sd = kv.pool_desc(src_c, src_r, 64, f["heads"], f["base"], pair_convention=f["il"])
        dd = kv.pool_desc(dst_c, dst_r, 64, f["heads"], f["base"], pair_convention=f["il"])
        dev = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).cuda()
               for k in ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta",
                         "block_tables")}
        ws = kv.workspace(dd, wl.total_tokens, wl.num_chunks)

        def call():
            kv.kv_relocate(sd, dd, wl.num_chunks, wl.total_tokens, dev["tok_off"],
                           dev["src_slots"], dev["chunk_req"], dev["chunk_dst_pos"],
                           dev["delta"], dev["block_tables"], wl.block_tables.shape[0],
                           wl.block_tables.shape[1], None, ws)
            return kv.kv_last_launch_count()

        barrier(world)
        ms, kms, n_l = _timed(call, K, W)
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        launches += n_l
        nbytes = wl.total_tokens * (L * 2 * 2 * (f["copy_dim"] + rw) + 4)
        entry = {"family": f["name"], "layers": L, "row_bf16": f["copy_dim"] + rw,
                 "pairs": "interleaved" if f["il"] else "rotate-half",
                 "tokens": wl.total_tokens, "kernel_ms": kms,
                 "achieved_gbs": nbytes / (kms * 1e-3) / 1e9,
                 "frac": nbytes / (kms * 1e-3) / 1e9 / peak, "algorithmic_bytes": nbytes}
        if orc is not None:
            entry["parity_sample"] = check_family_sample(f, wl, src_c, src_r, dst_c, dst_r, orc)
        res.append(entry)
        tot_tok += wl.total_tokens * world
        tot_ms += max_over_ranks(ms, world)
        if main is None or nbytes > main["algorithmic_bytes"]:
            main = entry
        del src_c, src_r, dst_c, dst_r, ws, dev
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    clk = clocks.stop()
    out = {
        "metric": "relocated KV tokens/s (all layers)",
        "value": tot_tok / (tot_ms * 1e-3), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": tot_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "impl": "ours",
        "config": {"workload": "families: relocation without a patch for "
                               + ", ".join(e["family"] for e in res)
                               + " (one step = one relocation of each)",
                   "families": res, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (%.0f GB moved per step)"
                         % (sum(e["algorithmic_bytes"] for e in res) / 1e9)},
        "roofline": {"bound": "hbm", "achieved": main["achieved_gbs"], "peak": peak,
                     "unit": "GB/s", "frac": main["frac"], "peak_kind": peak_kind,
                     "traffic": recorded_traffic("families"),
                     "kernel": f"relocate_kernel ({main['family']})",
                     "kernel_ms": main["kernel_ms"],
                     "algorithmic_bytes_per_launch": main["algorithmic_bytes"]},
        "e2e": None, "clocks": clk, "gpu_launches": launches,
    }
    if orc is not None:
        agg = {}
        for e in res:
            for k2, v2 in e["parity_sample"].items():
                agg[k2] = agg.get(k2, 0) + v2
        out["parity_sample"] = agg
    return out


# ---------------------------------------------------------------------------
# Workload: Irminsul content-defined chunking of token streams
# ---------------------------------------------------------------------------

CDC_TOKENS = dict(num_streams=384, stream_len=131072, vocab=129280, shared_segments=64,
                  log_mean=8, gear_seed=0x1F2E3D4C5B6A7988, fp_seed=0)
# A small case of the same kernels (16 MB of tokens).
CDC_TOKENS_SMALL = dict(CDC_TOKENS, num_streams=32)


def build_cdc(rank: int, cfg, device: str = "cuda"):
    import position_independent_mla_gb300 as kv

    ts = synth.token_streams(5005 + 100 * rank, [cfg["stream_len"]] * cfg["num_streams"],
                             vocab=cfg["vocab"], shared_segments=cfg["shared_segments"])
    total = len(ts.tokens)
    host = {"off": torch.from_numpy(ts.stream_off).pin_memory(),
            "tok": torch.from_numpy(ts.tokens).pin_memory()}
    dev = {k: v.to(device) for k, v in host.items()}
    out = dict(ends=torch.empty(total, dtype=torch.int64, device=device),
               fps=torch.empty(total, dtype=torch.int64, device=device),
               cnt=torch.zeros(1, dtype=torch.int64, device=device))
    ws = torch.empty(kv.kv_cdc_workspace_size(total), dtype=torch.uint8, device=device)
    return dict(ts=ts, host=host, dev=dev, ws=ws, total=total, cfg=cfg,
                threshold=1 << (64 - cfg["log_mean"]), **out)


def cdc_call(st, dev=None, stream=None):
    import position_independent_mla_gb300 as kv

    d, c = dev if dev is not None else st["dev"], st["cfg"]
    kv.kv_cdc(st["ts"].num_streams, d["off"], st["total"], d["tok"], c["gear_seed"],
              st["threshold"], c["fp_seed"], st["total"], st["ends"], st["fps"], st["cnt"],
              st["ws"], stream=stream)
    return kv.kv_last_launch_count()


def check_cdc(st, orc) -> dict:
    """Full parity: every chunk end and fingerprint of the last call against
    the oracle run on the same streams."""
    c = st["cfg"]
    w_ends, w_fps, w_n = orc.cdc(st["ts"].stream_off, st["ts"].tokens, c["gear_seed"],
                                 st["threshold"], c["fp_seed"])
    n = int(st["cnt"].item())
    ends = st["ends"][:n].cpu().numpy()
    fps = st["fps"][:n].cpu().numpy().view(np.uint64)
    same = n == w_n
    return {"chunks": n, "oracle_chunks": int(w_n),
            "ends_differing": int(np.sum(ends != w_ends)) if same else n,
            "fingerprints_differing": int(np.sum(fps != w_fps)) if same else n}


def run_cdc_tokens(args, rank, world, local):
    """Content-defined chunking of agentic token streams (Irminsul §2.2): every
    stream cut where its 64-token Gear hash falls below the threshold, every
    chunk fingerprinted with XXH64 -- four kernels per call."""
    import position_independent_mla_gb300 as kv

    cfg = CDC_TOKENS_SMALL if args.small else CDC_TOKENS
    st = build_cdc(rank, cfg)
    K, W = args.steps, args.warmup
    total = st["total"]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    ms, kms, launches = _timed(lambda: cdc_call(st), K, W)
    assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
    n_chunks = int(st["cnt"].item())
    # end to end: pinned host tokens and offsets in, the chunk count back
    host, dev = st["host"], st["dev"]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(K):
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        cdc_call(st, dev)
        n_back = int(st["cnt"].item())
        assert kv.kv_get_device_status(st["ws"], stream) == kv.KV_OK
    e2e_s = time.perf_counter() - t0
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(ms, world)
    e2e_s = max_over_ranks(e2e_s, world)
    nbytes = total * 4 + n_chunks * 16 + (st["ts"].num_streams + 1) * 8
    peak, peak_kind = hbm_peak()
    achieved = nbytes / (kms * 1e-3) / 1e9
    out = {
        "metric": "content-chunked tokens/s (Gear CDC + XXH64 fingerprints)",
        "value": total * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u64", "data": "synthetic", "impl": "ours",
        "config": {"workload": f"irminsul-cdc: {st['ts'].num_streams} token streams x "
                               f"{cfg['stream_len']} ids U[0,{cfg['vocab']}), each carrying "
                               f"segments of a {cfg['shared_segments']}-segment shared pool at "
                               "random offsets; Gear hash over 64-token windows, threshold "
                               f"2^{64 - cfg['log_mean']} (mean chunk {1 << cfg['log_mean']} "
                               "tokens), XXH64 per chunk",
                   "tokens_per_step_per_gpu": total, "chunks": n_chunks,
                   "mean_chunk_tokens": total / max(n_chunks, 1),
                   "parallelism": f"replicas x{world} (independent streams)",
                   "l2": "inputs larger than L2 (%.0f MB of token ids per step)" % (total * 4 / 1e6)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic("cdc_tokens"),
                     "kernel": "cdc_flags + cdc_scan + cdc_emit + fingerprint (whole call)",
                     "kernel_ms": kms, "algorithmic_bytes_per_step": nbytes},
        "e2e": {"value": total * world * K / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 8 + 4},
        "clocks": clk, "gpu_launches": launches,
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle as O
        orc = O.get()
        sample = synth.token_streams(77, [1 << 20] * 4, vocab=cfg["vocab"], shared_segments=8)
        t0 = time.perf_counter()
        orc.cdc(sample.stream_off, sample.tokens, cfg["gear_seed"], st["threshold"], cfg["fp_seed"])
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": len(sample.tokens) / dt, "unit": "tokens/s", "cores": 1,
                               "kind": "oracle",
                               "sample": f"4 streams x 2^20 tokens of the same recipe: {dt:.1f} s"}
    if args.check and rank == 0:
        import oracle as O
        out["parity_sample"] = check_cdc(st, O.get())
    return out


WORKLOADS = {"relocate-mla": run_relocate_mla, "splice-mla-128k": run_splice_mla_128k,
             "relocate-gqa-patch": run_relocate_gqa_patch, "splice-mla-4k": run_splice_mla_4k,
             "relocate-mla-patch": run_relocate_mla_patch, "sweep-mla": run_sweep_mla,
             "splice-mla-128k-composed": run_splice_mla_128k_composed,
             "splice-mla-128k-remap": run_splice_mla_128k_remap,
             "splice-mla-128k-remap-split":
                 lambda a, r, w, l: run_splice_mla_128k_remap(a, r, w, l, split=True),
             "window-gqa": run_window_gqa, "cdc-tokens": run_cdc_tokens,
             "families": run_families}


# The configured workloads, one JSON line each, the headline (the Irminsul
# MLA relocation) last: the 4096-token splice, the 128K-context splice, the
# Kamera GQA relocation with its fused rank-16 patch, the MLA sweep.
DEFAULT_SEQUENCE = ("splice-mla-4k", "splice-mla-128k", "relocate-gqa-patch", "sweep-mla",
                    "relocate-mla")
SWEEP_MAX_STEPS = 10   # per sweep point in the default sequence (41 points)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=160)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["default"] + sorted(WORKLOADS), default="default",
                    help="default: every configured workload, one line each, the headline "
                         "relocation last")
    ap.add_argument("--check", action="store_true", help="sampled parity vs the oracle")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true",
                    help="a reduced batch of the same workload (for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_info()

    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    import position_independent_mla_gb300 as kv

    kv.load()  # raises if the CUDA library is missing: there is no fallback
    names = DEFAULT_SEQUENCE if args.workload == "default" else (args.workload,)
    cores = None
    if rank == 0 and not args.no_cpu_baseline and any(n in CPU_SAMPLES for n in names):
        cores = OracleCores()   # spawned processes, one per host core
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        for name in names:
            wargs = args
            if name == "sweep-mla" and len(names) > 1:
                wargs = argparse.Namespace(**dict(vars(args), steps=min(args.steps,
                                                                       SWEEP_MAX_STEPS)))
            out = WORKLOADS[name](wargs, rank, world, local)
            gc.collect()
            torch.cuda.empty_cache()   # the next workload gets the whole HBM
            if args.small and isinstance(out.get("roofline"), dict):
                # the recorded DRAM traffic is that of the full workload
                out["roofline"]["traffic"] = None
            if cores is not None and name in CPU_SAMPLES:
                out["cpu_baseline"] = cpu_baseline(name, out["unit"], cores)
            if rank == 0:
                print(json.dumps(add_nominal(out)), flush=True)
            barrier(world)
    finally:
        if cores is not None:
            cores.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
