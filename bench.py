"""Decode-step benchmark of the paged K/V-cache path on GB300.

One step = one decode step of the OPT-13B-shaped single-layer batch (64
sequences, 40 heads x 128, block size 16, context lengths ~ U[128, 2048],
physical blocks shuffled): copy_blocks of the step's copy-on-write pairs,
reshape_and_cache of the 64 new tokens, paged decode attention (partition
kernel + merge kernel).  Slot assignment (the host block manager) runs once
at set-up; its host time is reported separately.

Prints ONE JSON line (rank 0).  `value` is effective KV GB/s: the K/V bytes
attention reads per step (logical, a shared block counted per reader) over
the device-timed step.  `e2e` is the same metric through the same C-ABI
calls with every step's inputs in page-locked host memory, read by the kernels
across NVLink-C2C, and the output written back there (`staged_value`: the
same step with one host->device and one device->host copy).  `roofline` is
the paged attention call alone against the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload opt13b|parallel_sampling|parallel_sampling_cow|shared_prefix|capacity|beam_search
                              |swap|layers40|prefill]
                  [--capacity-seqs S] [--capacity-block B] [--pool-frac F] [--grouped]

`--workload swap`, `--workload layers40` and `--workload prefill` print their
own lines (swap_blocks between HBM and page-locked host memory; 40-layer
copy_blocks and reshape_and_cache in one launch; prefill attention over a
cached prefix on the tensor cores) with their own metric names.

The default workload is the headline one above.  The others build their batch
through the same block manager (prompt forks with copy-on-write, a shared
prefix, full 2048-token contexts); their copy-on-write copies are timed as
one copy_blocks call (`copy_blocks_setup`).

--grouped makes the attention call pkv_paged_attention_decode_shared_prefix:
consecutive sequences whose leading blocks are the same physical blocks form a
group whose shared prefix is read once (groups under 8 members still read it
per sequence); the metric is unchanged and `roofline` then counts distinct K/V
slots.

--impl reference times the CPU oracle on the host cores instead (a bounded
sample of the same workload per step) and prints the same metric.
"""
from __future__ import annotations

import argparse
import atexit
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

# the CPU baseline's "one core" must be one: numpy's BLAS would otherwise spread matrix products
# over every core (set before numpy loads; the all-cores figure uses one process per core)
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention effective KV GB/s (% of HBM peak) and decode tokens/s"
UNIT = "GB/s"
WORKLOAD = ("opt13b_decode_step: 64 seqs, 40 heads x 128, block 16, ctx ~ U[128,2048], shuffled blocks, "
            "+ the K/V write of 64 new tokens (in the attention launch; --unfused: reshape_and_cache first)")
SEED = 1002
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0                                # GB300 HBM3e, nominal
EVENT_EVERY = 16

# dram__bytes_read.sum + dram__bytes_write.sum of one paged-attention call (partition + merge
# kernels) from an ncu capture, keyed by (workload, sha256 of the attention source it was taken
# on); a changed kernel reports null until it is captured again.
NCU_TRAFFIC = {
    # the headline step's fused call: partition kernel 1,373,092,500 B read + 4,835,200 B written
    # (the appended rows included), merge kernel 1,280,000 B read (means of two launches each;
    # profiles/paged_attention_opt13b_decode.md; captured on source 671088f0..., which differs from
    # this key's source in the file's header comment only)
    ("opt13b+append", "5db4ea62901c2074d5db6247fb9ca0f86ae177cb2d1f094b6e25a2b6456c7857"): 1_379_208_000,
}


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer loop (profiling runs)")
    ap.add_argument("--unfused", action="store_true",
                    help="write the new tokens with a separate reshape_and_cache call before attention "
                         "(default: pkv_paged_attention_decode_append, one launch)")
    ap.add_argument("--grouped", action="store_true",
                    help="read each shared prefix once per group of sequences (shared-prefix decode entry); "
                         "groups come from the block manager's shared leading blocks")
    ap.add_argument("--workload", choices=WORKLOADS + AUX_WORKLOADS, default="opt13b",
                    help="opt13b (the headline batch) or another decode batch of the same shape family")
    ap.add_argument("--capacity-seqs", type=int, default=64, help="capacity workload: sequences (ctx 2048 each)")
    ap.add_argument("--capacity-block", type=int, default=16, help="capacity workload: block size")
    ap.add_argument("--pool-frac", type=float, default=0.0,
                    help="capacity workload: size the pool to this fraction of free HBM (0 = just enough)")
    return ap.parse_args()


def attention_source_sha() -> str:
    path = os.path.join(ROOT, "paged_kv_cache_73_gb300", "csrc", "attention.cu")
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: torch copy, read+write bytes)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms by a child process.

    The sampler starts before the warm-up steps and runs until the run ends. Each sample carries
    nvidia-smi's own timestamp. `summary(t0, t1)` keeps the samples whose timestamps fall inside the
    timed region [t0, t1] (host wall clock). When the region is shorter than three intervals it also
    keeps the last sample before t0 and the first after t1; the warm-up keeps the GPU busy before."""

    INTERVAL_MS = 100
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.out = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="pkv_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        if self.out is not None:
            self.out.close()
            self.out = None
        if self.path is not None and os.path.exists(self.path):
            os.unlink(self.path)

    def __enter__(self):
        return self.start()

    def __exit__(self, *exc):
        self.stop()

    @staticmethod
    def _stamp(text):
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                continue
        return None

    def _rows(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 10:
                        rows.append((self._stamp(parts[0]), parts))
        except OSError:
            pass
        return rows

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return None
        # wait (bounded) for the first sample after the region
        deadline = time.time() + 1.0
        rows = self._rows()
        while time.time() < deadline and not any(t is not None and t > t1 for t, _ in rows):
            time.sleep(0.05)
            rows = self._rows()
        if not rows:
            return None
        stamped = [(t, r) for t, r in rows if t is not None]
        if stamped:
            inside = [r for t, r in stamped if t0 <= t <= t1]
            window = "inside the timed region"
            if len(inside) < 3:
                before = [r for t, r in stamped if t < t0][-1:]
                after = [r for t, r in stamped if t > t1][:1]
                inside = before + inside + after
                window = "inside the timed region, plus the last sample before it and the first after it"
            picked = inside
        else:
            picked = [r for _, r in rows]
            window = "unparsed timestamps: every sample since the sampler started"
        if not picked:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in picked if num(r[2]) is not None]
        reasons = set()
        for r in picked:
            for name, val in zip(self.REASONS, r[6:10]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": num(picked[0][3]), "samples": len(picked), "interval_ms": self.INTERVAL_MS,
                "window": window, "region_s": t1 - t0,
                "power_w_max": max((num(r[4]) or 0.0) for r in picked), "reasons": sorted(reasons)}


# ---- workloads -------------------------------------------------------------------------------------

WORKLOADS = ("opt13b", "parallel_sampling", "parallel_sampling_cow", "shared_prefix", "capacity", "beam_search")


def attention_algorithmic_bytes(w) -> int:
    """K/V rows read + q read + out written + table entries + context lengths, per call."""
    H, D, B = w.num_heads, w.head_dim, w.block_size
    total = 0
    for c in w.context_lens:
        c = int(c)
        total += H * (2 * c * D * 2 + 2 * D * 2) + 4 * math.ceil(c / B) + 4
    return total


def shared_prefix_groups(tables, lens, B):
    """Groups of consecutive sequences whose leading blocks are the same physical blocks (the block
    manager's shared prompt or prefix) and each group's shared whole-block prefix length."""
    S = len(lens)
    starts, prefixes = [0], []
    s = 0
    while s < S:
        e = s + 1
        while e < S and tables[e, 0] == tables[s, 0]:
            e += 1
        nb = 0
        if e - s > 1:
            cap = min(int(lens[i]) for i in range(s, e)) // B      # blocks full in every member
            while nb < cap and all(tables[i, nb] == tables[s, nb] for i in range(s + 1, e)):
                nb += 1
        prefixes.append(nb * B)
        starts.append(e)
        s = e
    return np.array(starts, dtype=np.int32), np.array(prefixes, dtype=np.int32)


def _grow(bm, seqs, targets):
    """Append tokens to `seqs` until each holds targets[i] - 1 tokens; returns the copies made."""
    copies = []
    have = {s: bm.block_table(s)[1] for s in seqs}
    while True:
        live = [s for s, t in zip(seqs, targets) if have[s] < t - 1]
        if not live:
            return copies
        _, pairs = bm.append_slots(live)
        copies += [tuple(int(x) for x in p) for p in pairs]
        for s in live:
            have[s] += 1


def block_manager_summary(bm) -> dict:
    """The manager's state after the step's slot assignment: occupancy, sharing and events."""
    free, waste, _ = bm.stats()
    return {"free_blocks": free, "tail_waste_tokens": waste, "ref_histogram": bm.ref_histogram(8).tolist(),
            **bm.counters()}


def build_step_inputs(seed: int, workload: str = "opt13b", capacity_seqs: int = 64, capacity_block: int = 16,
                      pool_blocks=None):
    """A decode step's batch built through the host block manager over the recipe's lengths.

    Every sequence is grown to ctx - 1 tokens (prefill, forks, copy-on-write and
    earlier decode tokens as the workload prescribes), then one append per
    sequence gives this step's new-token slots and copy pairs.
    Returns a dict: w (DecodeWorkload over the manager's tables), slots, pairs
    (this step's copies), setup_pairs (copies made while growing), host_us,
    desc.
    """
    from paged_kv_cache_73_gb300 import binding as pkv
    from paged_kv_cache_73_gb300 import workloads as wl

    if workload == "beam_search":
        return build_beam_step(seed)
    if workload == "opt13b":
        recipe = wl.opt13b(seed=seed)
    elif workload in ("parallel_sampling", "parallel_sampling_cow"):
        recipe = wl.parallel_sampling(seed=seed, prompt_len=512 if workload == "parallel_sampling" else 511)
    elif workload == "shared_prefix":
        recipe = wl.shared_prefix(seed=seed)
    elif workload == "capacity":
        recipe = wl.capacity(seed=seed, num_seqs=capacity_seqs, block_size=capacity_block, num_blocks=pool_blocks)
    else:
        raise ValueError(workload)
    H, D, B = recipe.num_heads, recipe.head_dim, recipe.block_size
    lens = recipe.context_lens
    S = len(lens)
    N = recipe.num_blocks
    bm = pkv.BlockManager(N, B, wl.free_list_order(N, seed))
    seqs = list(range(S))
    setup = []
    if workload.startswith("parallel_sampling"):
        n, prompt = 4, 512 if workload == "parallel_sampling" else 511
        for base in range(0, S, n):
            bm.add_seq(base, prompt)
            for i in range(1, n):
                bm.fork(base, base + i)
        setup = _grow(bm, seqs, lens)
    elif workload == "shared_prefix":
        bm.register_prefix(0, 1024)
        for s in seqs:
            bm.add_seq_with_prefix(s, 0)
        setup = _grow(bm, seqs, lens)
    else:
        for s in seqs:
            bm.add_seq(s, int(lens[s]) - 1)
    t0 = time.perf_counter()
    slots, pairs = bm.append_slots(seqs)                # slot assignment of this step's token
    host_us = (time.perf_counter() - t0) * 1e6
    max_blocks = -(-2048 // B) if workload == "opt13b" else -(-int(lens.max()) // B)
    tables, ctx = bm.block_tables(seqs, max_blocks)
    assert np.array_equal(ctx, lens)
    w = wl.from_tables(f"{workload}_decode_step", seed, H, D, B, N, tables, ctx, recipe.notes)
    if workload == "capacity":
        desc = f"capacity: {S} seqs x ctx 2048, 40 x 128, block {B}, {N} pool blocks, shuffled"
    elif workload == "opt13b":
        desc = WORKLOAD
    else:
        desc = f"{workload}: {recipe.notes}, 40 x 128, block {B}, shuffled blocks"
    return {"w": w, "slots": slots, "pairs": pairs, "setup_pairs": np.array(setup, dtype=np.int64).reshape(-1, 2),
            "host_us": host_us, "desc": desc, "workload": workload, "bm": block_manager_summary(bm)}


def build_beam_step(seed: int, requests: int = 16, width: int = 4, beam_steps: int = 128, B: int = 16):
    """Beam search through the block manager: each request keeps `width` candidates; every step
    each new candidate picks a parent among the current ones (seeded), the old beam is retired and
    shared partly filled blocks are copied once per extra sibling.  The measured step is one more
    beam step: its copies, its new tokens' writes and attention over all candidates."""
    from paged_kv_cache_73_gb300 import binding as pkv
    from paged_kv_cache_73_gb300 import workloads as wl

    H, D = 40, 128
    rng = np.random.default_rng(seed)
    prompts = rng.integers(256, 1025, size=requests)
    N = int(2 * (sum(-(-int(p) // B) for p in prompts) + requests * width * (beam_steps // B + 3)))
    bm = pkv.BlockManager(N, B, wl.free_list_order(N, seed))
    beams, nid = [], 0
    for r in range(requests):
        bm.add_seq(nid, int(prompts[r]))
        beams.append([nid])
        nid += 1
    setup = []

    def one_step():
        nonlocal nid
        slots, pairs = [], []
        for r in range(requests):
            parents = [int(x) for x in rng.choice(beams[r], size=width)]
            children = list(range(nid, nid + width))
            nid += width
            sl, pr = bm.beam_step(parents, children, beams[r])
            beams[r] = children
            slots += [int(x) for x in sl]
            pairs += [tuple(int(y) for y in p) for p in pr]
        return slots, pairs

    for _ in range(beam_steps):
        setup += one_step()[1]
    t0 = time.perf_counter()
    slots, pairs = one_step()
    host_us = (time.perf_counter() - t0) * 1e6
    seqs = [c for beam in beams for c in beam]
    lens = np.array([bm.block_table(c)[1] for c in seqs], dtype=np.int32)
    max_blocks = -(-int(lens.max()) // B)
    tables, ctx = bm.block_tables(seqs, max_blocks)
    w = wl.from_tables("beam_search_decode_step", seed, H, D, B, N, tables, ctx,
                       f"{requests} requests x beam width {width}, prompts U[256,1024], {beam_steps} beam steps")
    desc = f"beam_search: {w.notes}, 40 x 128, block {B}, shuffled blocks"
    return {"w": w, "slots": np.array(slots, dtype=np.int64),
            "pairs": np.array(pairs, dtype=np.int64).reshape(-1, 2),
            "setup_pairs": np.array(setup, dtype=np.int64).reshape(-1, 2), "host_us": host_us, "desc": desc,
            "workload": "beam_search", "bm": block_manager_summary(bm)}


def run_gpu(args, rank, world, dev):
    import torch
    from paged_kv_cache_73_gb300 import binding as pkv
    from paged_kv_cache_73_gb300 import workloads as wl

    seed = SEED + 7919 * rank                           # weak scaling: each rank its own batch
    x = build_step_inputs(seed, args.workload, args.capacity_seqs, args.capacity_block,
                          pool_blocks_for(args, dev))
    w, slots, pairs = x["w"], x["slots"], x["pairs"]
    S, H, D, B, MB = w.num_seqs, w.num_heads, w.head_dim, w.block_size, w.max_blocks_per_seq
    k, v = w.pools(dev)
    q = w.q(dev)
    key, value = wl.new_tokens(S, H, D, seed, dev)
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    slots_d = torch.from_numpy(slots).to(dev)
    pairs_d = torch.from_numpy(np.ascontiguousarray(pairs)).to(dev)
    out = torch.empty_like(q)
    ws = pkv.workspace_for(S, H, D, MB, B, dev)
    part_tokens, attn_kernels = pkv.paged_attention_plan(S, H, D, MB, B)
    stream = torch.cuda.current_stream()
    n_pairs = int(pairs.shape[0])
    grouped = None
    if args.grouped:
        gs_h, pl_h = shared_prefix_groups(w.block_tables, w.context_lens, B)
        n_ws = pkv.paged_attention_shared_prefix_workspace_size(S, H, D, MB, B)
        grouped = {"gs": torch.from_numpy(gs_h).to(dev), "pl": torch.from_numpy(pl_h).to(dev),
                   "max_group": int(np.max(np.diff(gs_h))), "groups": int(len(pl_h)),
                   "prefix_tokens": int(pl_h.sum()), "gs_h": gs_h, "pl_h": pl_h}
        ws = torch.empty(max(n_ws, 16), dtype=torch.uint8, device=dev)
        attn_kernels = 3                                 # prefix partials, partitions, merge

    def attention(qq, tt, ll, st):
        if grouped is None:
            pkv.paged_attention_decode(qq, k, v, tt, ll, w.scale, B, out=out, workspace=ws, stream=st)
        else:
            pkv.paged_attention_decode_shared_prefix(qq, k, v, tt, ll, grouped["gs"], grouped["pl"], w.scale, B,
                                                     grouped["max_group"], out=out, workspace=ws, stream=st)

    copy = None
    if len(x["setup_pairs"]):
        # the copy-on-write copies made while the batch grew, as one copy_blocks call
        sp = torch.from_numpy(np.ascontiguousarray(x["setup_pairs"])).to(dev)
        for _ in range(5):
            pkv.copy_blocks([k], [v], sp, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(20):
            pkv.copy_blocks([k], [v], sp, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / 20
        moved = 2 * 2 * len(sp) * H * B * D * 2           # K and V, read and written
        copy = {"pairs": int(len(sp)), "ms": ms, "GB/s": moved / (ms * 1e-3) / 1e9}

    fused = grouped is None and not args.unfused

    def step(ev0=None, ev1=None):
        if n_pairs:
            pkv.copy_blocks([k], [v], pairs_d, stream=stream)
        if fused:
            # the new tokens' K/V write and the attention in one launch
            if ev0 is not None:
                ev0.record(stream)
            pkv.paged_attention_decode_append(q, key, value, slots_d, k, v, tables, lens, w.scale, B, out=out,
                                              workspace=ws, stream=stream)
        else:
            pkv.reshape_and_cache(key, value, k, v, slots_d, stream=stream)
            if ev0 is not None:
                ev0.record(stream)
            attention(q, tables, lens, stream)
        if ev1 is not None:
            ev1.record(stream)

    # clocks sampled from before the warm-up on; stopped at exit as well, should the run raise
    clocks = ClockSampler(physical_gpu_index(torch.cuda.current_device())).start()
    atexit.register(clocks.stop)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0

    K = args.steps
    l2_bytes = l2_cache_bytes(dev)
    flush = w.physical_kv_bytes() < 2 * l2_bytes
    barrier(world)
    torch.cuda.synchronize()
    if flush:
        # a step whose K/V would stay in L2: a write of twice the L2 size before every step, outside
        # the timed region, and each step timed by its own events (start, attention, end)
        scratch = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
        t0 = time.time()
        for i in range(K):
            scratch.fill_(i & 255)
            e0, e1, e2 = evs[i]
            e0.record(stream)
            step(e1, e2)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        step_ms = sum(e0.elapsed_time(e2) for e0, _, e2 in evs) / K
        attn_ms = [e1.elapsed_time(e2) for _, e1, e2 in evs]
    else:
        # events around the attention call on every EVENT_EVERY-th step only: an event between two
        # kernels stops the next launch from overlapping the previous kernel's tail (PDL)
        n_ev = (K + EVENT_EVERY - 1) // EVENT_EVERY
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        start.record(stream)
        for i in range(K):
            if i % EVENT_EVERY == 0:
                step(*ev[i // EVENT_EVERY])
            else:
                step()
        stop.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        step_ms = start.elapsed_time(stop) / K
        attn_ms = [a.elapsed_time(b) for a, b in ev]
    clock_summary = clocks.summary(t0, t1)
    clocks.stop()
    code = pkv.device_error()
    assert code == 0, f"device check {code}"

    res = {"step_ms": step_ms, "attn_ms": sum(attn_ms) / len(attn_ms), "attn_ms_median": statistics.median(attn_ms),
           "l2_flushed": flush,
           "kv_bytes": w.logical_kv_bytes(), "phys_bytes": w.physical_kv_bytes(),
           # grouped: each shared prefix is read once, so the call's bytes are the distinct slots;
           # fused: the call also reads the new K/V rows and writes them into the pools
           "attn_bytes": (attention_algorithmic_bytes(w) + (4 * S * H * D * 2 if fused else 0)) if grouped is None
           else w.physical_kv_bytes() + S * H * D * 2 * 2,
           "fused": fused,
           "grouped": None if grouped is None else {k_: grouped[k_] for k_ in ("groups", "max_group", "prefix_tokens")},
           "num_seqs": S,
           "launches": K * ((1 if n_pairs else 0) + (0 if fused else 1) + attn_kernels), "part_tokens": part_tokens,
           "host_slot_us": x["host_us"], "clocks": clock_summary, "n_pairs": n_pairs, "copy": copy,
           "desc": x["desc"], "num_blocks": w.num_blocks, "bm": x["bm"]}
    if not args.no_e2e:
        res.update(run_e2e(args, w, slots, pairs, q, key, value, k, v, dev, ws, grouped, fused))
    return res


AUX_WORKLOADS = ("swap", "layers40", "prefill")


def _timed(fn, reps=10, warm=3):
    import torch
    for _ in range(warm):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _timed_graph(fn, reps=20, warm=3):
    """Device time of fn's launches: captured once as a CUDA graph and replayed, so the host's
    per-call argument marshalling (a pointer per layer and pool) does not pace the GPU."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    for _ in range(warm):
        g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_swap(args, dev):
    """swap_blocks: the blocks of 16 sequences x 2048 tokens (one layer, 40 x 128, block 16)
    out to page-locked host memory and back, one launch each way, against one
    cudaMemcpyAsync per block (the pattern the fused kernel replaces)."""
    import torch
    from paged_kv_cache_73_gb300 import binding as pkv
    from paged_kv_cache_73_gb300 import workloads as wl
    H, D, B, n = 40, 128, 16, 16 * 128
    N = n + 512
    dk = wl.dense_tensor((N, H, B, D), SEED, wl.STREAM_K, dev)
    dv = wl.dense_tensor((N, H, B, D), SEED, wl.STREAM_V, dev)
    hk = torch.empty((n, H, B, D), dtype=torch.float16, pin_memory=True)
    hv = torch.empty_like(hk).pin_memory()
    rng = np.random.default_rng(SEED)
    src = rng.permutation(N)[:n]
    out_map = torch.from_numpy(np.stack([src, np.arange(n)], 1).astype(np.int64)).to(dev)
    back = rng.permutation(np.setdiff1d(np.arange(N), src))
    spare = np.concatenate([back, src])[:n]
    in_map = torch.from_numpy(np.stack([np.arange(n), spare], 1).astype(np.int64)).to(dev)
    payload = 2 * n * H * B * D * 2                          # K and V bytes moved each way
    t_out = _timed(lambda: pkv.swap_blocks([dk], [dv], [hk], [hv], out_map))
    t_in = _timed(lambda: pkv.swap_blocks([hk], [hv], [dk], [dv], in_map))
    assert pkv.device_error() == 0
    ok = torch.equal(dk[torch.from_numpy(spare).to(dev)].cpu(), hk)
    src_l, spare_l = src.tolist(), spare.tolist()

    def per_block_out():
        for i, s_ in enumerate(src_l):
            hk[i].copy_(dk[s_], non_blocking=True)
            hv[i].copy_(dv[s_], non_blocking=True)

    def per_block_in():
        for i, d_ in enumerate(spare_l):
            dk[d_].copy_(hk[i], non_blocking=True)
            dv[d_].copy_(hv[i], non_blocking=True)

    m_out = _timed(per_block_out, reps=3, warm=1)
    m_in = _timed(per_block_in, reps=3, warm=1)
    gbs = lambda ms: payload / (ms * 1e-3) / 1e9
    value = 2 * payload / ((t_out + t_in) * 1e-3) / 1e9
    return {"metric": "swap_blocks GB/s (HBM <-> page-locked Grace memory, both directions)", "value": value,
            "unit": "GB/s", "n_gpus": 1, "higher_is_better": True, "dtype": "f16 (bit copy)",
            "data": "synthetic (seeded counter-based generator)", "round_trip_bit_exact": bool(ok),
            "config": {"workload": "swap: 2048 blocks (16 seqs x 2048 tokens), 40 x 128, block 16, one layer",
                       "bytes_each_way": payload},
            "swap_out": {"ms": t_out, "GB/s": gbs(t_out), "launches": 1},
            "swap_in": {"ms": t_in, "GB/s": gbs(t_in), "launches": 1},
            "per_block_memcpy": {"out_ms": m_out, "in_ms": m_in, "out_GB/s": gbs(m_out), "in_GB/s": gbs(m_in),
                                 "copies_each_way": 2 * n}}


def run_layers40(args, dev):
    """The OPT-13B layer count: reshape_and_cache of 64 tokens and 96 copy-on-write copies over 40
    layers, each as one launch, against one launch per layer."""
    import torch
    from paged_kv_cache_73_gb300 import binding as pkv
    H, D, B, N, L, T = 40, 128, 16, 1024, 40, 64
    ks = [torch.zeros((N, H, B, D), dtype=torch.float16, device=dev) for _ in range(L)]
    vs = [torch.zeros((N, H, B, D), dtype=torch.float16, device=dev) for _ in range(L)]
    keys = [torch.ones((T, H, D), dtype=torch.float16, device=dev) for _ in range(L)]
    vals = [torch.ones((T, H, D), dtype=torch.float16, device=dev) for _ in range(L)]
    rng = np.random.default_rng(SEED)
    slots = torch.from_numpy(rng.choice(N * B, size=T, replace=False).astype(np.int64)).to(dev)
    perm = rng.permutation(N)
    pairs = torch.from_numpy(np.stack([perm[:96], perm[96:192]], 1).astype(np.int64)).to(dev)
    # device time (graph replay of the same calls), and the eager call time with the host's work
    t_r1 = _timed_graph(lambda: pkv.reshape_and_cache_layers(keys, vals, ks, vs, slots), reps=50)
    t_rL = _timed_graph(lambda: [pkv.reshape_and_cache(keys[l], vals[l], ks[l], vs[l], slots) for l in range(L)],
                        reps=50)
    t_c1 = _timed_graph(lambda: pkv.copy_blocks(ks, vs, pairs), reps=20)
    t_cL = _timed_graph(lambda: [pkv.copy_blocks([ks[l]], [vs[l]], pairs) for l in range(L)], reps=20)
    e_r1 = _timed(lambda: pkv.reshape_and_cache_layers(keys, vals, ks, vs, slots), reps=50)
    e_c1 = _timed(lambda: pkv.copy_blocks(ks, vs, pairs), reps=20)
    assert pkv.device_error() == 0
    r_bytes = 2 * 2 * L * T * H * D * 2                      # K and V, read and written
    c_bytes = 2 * 2 * L * 96 * H * B * D * 2
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9
    return {"metric": "multi-layer cache ops GB/s (40 layers, one launch)", "value": gbs(c_bytes, t_c1),
            "unit": "GB/s", "n_gpus": 1, "higher_is_better": True, "dtype": "f16 (bit copy)", "data": "synthetic",
            "config": {"workload": "layers40: 40 layers x [1024 blocks, 40, 16, 128]; 64 new tokens; 96 copy pairs"},
            "timing": "device time of CUDA-graph replays of the calls; eager_call_ms adds the host's argument "
                      "marshalling (one pointer per layer and pool)",
            "copy_blocks": {"one_launch_ms": t_c1, "one_launch_GB/s": gbs(c_bytes, t_c1),
                            "per_layer_launches_ms": t_cL, "per_layer_GB/s": gbs(c_bytes, t_cL),
                            "eager_call_ms": e_c1},
            "reshape_and_cache": {"one_launch_ms": t_r1, "one_launch_GB/s": gbs(r_bytes, t_r1),
                                  "per_layer_launches_ms": t_rL, "per_layer_GB/s": gbs(r_bytes, t_rL),
                                  "eager_call_ms": e_r1}}


def run_prefill(args, dev):
    """Prefill over a cached prefix: the shared-prefix batch (256 requests, one cached 1024-token
    prefix, suffixes U[32, 512]) writes every suffix token's K/V (reshape_and_cache) and runs
    paged prefill attention for the suffix tokens over prefix + causal suffix."""
    import torch
    from paged_kv_cache_73_gb300 import binding as pkv
    from paged_kv_cache_73_gb300 import workloads as wl
    w = wl.shared_prefix(seed=SEED)
    H, D, B = w.num_heads, w.head_dim, w.block_size
    news = np.array([int(c) - 1024 for c in w.context_lens])
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    T = int(qs[-1])
    slots = []
    for s_, (c, n) in enumerate(zip(w.context_lens, news)):
        for pos in range(int(c) - int(n), int(c)):
            slots.append(int(w.block_tables[s_, pos // B]) * B + pos % B)
    k, v = w.pools(dev)
    q = wl.dense_tensor((T, H, D), SEED, wl.STREAM_Q, dev)
    key, value = wl.new_tokens(T, H, D, SEED, dev)
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    qsd = torch.from_numpy(qs).to(dev)
    slots_d = torch.tensor(slots, dtype=torch.int64, device=dev)
    out = torch.empty_like(q)
    maxq = int(news.max())
    flops = sum(4 * D * H * int((np.arange(int(c) - int(n), int(c)) + 1).sum()) for c, n in zip(w.context_lens, news))
    attn = lambda: pkv.paged_attention_prefill(q, k, v, tables, lens, qsd, w.scale, B, maxq, out=out)

    def step():
        pkv.reshape_and_cache(key, value, k, v, slots_d)
        attn()

    # long prompts with nothing cached: 8 x 4096 tokens, causal over themselves
    wl2 = wl.custom(SEED + 5, [4096] * 8, H, D, B, name="prefill_8x4096")
    k2, v2 = wl2.pools(dev)
    qs2 = np.arange(0, 8 * 4096 + 1, 4096, dtype=np.int32)
    q2 = wl.dense_tensor((8 * 4096, H, D), SEED + 1, wl.STREAM_Q, dev)
    out2 = torch.empty_like(q2)
    t2, l2, qs2d = (torch.from_numpy(x).to(dev) for x in (wl2.block_tables, wl2.context_lens, qs2))
    flops2 = 8 * 4 * D * H * (4096 * 4097 // 2)
    attn2 = lambda: pkv.paged_attention_prefill(q2, k2, v2, t2, l2, qs2d, wl2.scale, B, 4096, out=out2)

    steps = max(3, min(args.steps, 50))
    with ClockSampler(physical_gpu_index(torch.cuda.current_device())) as clocks:
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        t0 = time.time()
        t_step = _timed(step, reps=steps, warm=max(args.warmup, 3))
        t_attn = _timed(attn, reps=steps, warm=3)
        t_long = _timed(attn2, reps=steps, warm=3)
        t1 = time.time()
        clock_summary = clocks.summary(t0, t1)
    assert pkv.device_error() == 0
    peak = measured_tensor_peak()
    achieved = flops / (t_attn * 1e-3) / 1e12
    return {"metric": "paged prefill attention TFLOP/s (new tokens over cached prefix + causal suffix)",
            "value": flops / (t_step * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": steps,
            "warmup": max(args.warmup, 3), "ms_per_step": t_step, "higher_is_better": True, "dtype": "f16 in, f32 acc",
            "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": "prefill: 256 requests, cached 1024-token prefix (shared blocks), suffixes "
                                   "U[32,512] prefilled; 40 x 128, block 16", "new_tokens": T,
                       "attention_flops": flops},
            "tokens_per_s": T / (t_step * 1e-3),
            "long_prompts": {"workload": "8 x 4096-token prompts, nothing cached, causal; 40 x 128, block 16",
                             "ms": t_long, "TFLOP/s": flops2 / (t_long * 1e-3) / 1e12,
                             "tokens_per_s": 8 * 4096 / (t_long * 1e-3), "frac": flops2 / (t_long * 1e-3) / 1e12 / peak[0]},
            "roofline": {"bound": "tensor", "kernel": "paged_prefill_tc_kernel", "achieved": achieved,
                         "peak": peak[0], "unit": "TFLOP/s", "frac": achieved / peak[0], "traffic": None,
                         "launch_ms": t_attn, "peak_source": peak[1]},
            "clocks": clock_summary}


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured bf16 dense burst (MEASURED_PEAKS.json bf16_tflops; fp16 has the same nominal rate), of measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback 1.9 PFLOP/s bf16 burst"


def pool_blocks_for(args, dev):
    """Pool size for the capacity workload: a fraction of free HBM, or just enough."""
    if args.workload != "capacity" or args.pool_frac <= 0:
        return None
    import torch
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info(dev)
    per_block = 2 * 40 * args.capacity_block * 128 * 2
    return int(args.pool_frac * free / per_block)


def physical_gpu_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    if local < len(ids) and ids[local].isdigit():
        return int(ids[local])
    return local


def run_e2e(args, w, slots, pairs, q, key, value, k, v, dev, ws, grouped=None, fused=False):
    """Same step through the C ABI, with the step's inputs in pinned host memory, two ways.

    direct: the kernels read q, the new keys/values, slot mapping, copy pairs,
    block tables and context lengths from the page-locked host buffer across the
    host link (NVLink-C2C) and write the attention output into page-locked host
    memory; the step ends when the stream has finished (wall clock).  Each step's
    1.4 GB K/V stream evicts the previous step's lines from L2, so every step's
    inputs cross the link again.
    staged: one packed host->device copy of the same inputs, the kernels, and a
    device->host copy of the output, then the wait.
    The shared-prefix entry loads q by TMA from device memory, so a grouped step
    is measured staged only.
    """
    import torch
    from paged_kv_cache_73_gb300 import binding as pkv

    parts = {
        "q": q.cpu(), "key": key.cpu(), "value": value.cpu(),
        "slots": torch.from_numpy(slots),
        "pairs": torch.from_numpy(np.ascontiguousarray(pairs)),
        "tables": torch.from_numpy(w.block_tables),
        "lens": torch.from_numpy(w.context_lens),
    }
    if grouped is not None:
        parts["gs"] = torch.from_numpy(grouped["gs_h"])
        parts["pl"] = torch.from_numpy(grouped["pl_h"])
    # one pinned byte buffer holding every input at a 256-byte-aligned offset, and its device twin
    offs, total = {}, 0
    for n, t in parts.items():
        offs[n] = total
        total += -(-(t.numel() * t.element_size()) // 256) * 256
    host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    dbuf, hbuf = {}, {}
    for n, t in parts.items():
        nbytes = t.numel() * t.element_size()
        host_buf[offs[n]:offs[n] + nbytes].copy_(t.contiguous().view(-1).view(torch.uint8))
        dbuf[n] = dev_buf[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)
        hbuf[n] = host_buf[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)
    out_h = torch.empty(tuple(q.shape), dtype=torch.float16).pin_memory()
    out_d = torch.empty_like(q)
    n_pairs = int(pairs.shape[0])
    h2d = sum(t.numel() * t.element_size() for t in parts.values())
    d2h = out_h.numel() * out_h.element_size()

    def step_calls(st, src, out):
        if n_pairs:
            pkv.copy_blocks([k], [v], src["pairs"], stream=st)
        if fused:
            pkv.paged_attention_decode_append(src["q"], src["key"], src["value"], src["slots"], k, v, src["tables"],
                                              src["lens"], w.scale, w.block_size, out=out, workspace=ws, stream=st)
            return
        pkv.reshape_and_cache(src["key"], src["value"], k, v, src["slots"], stream=st)
        if grouped is None:
            pkv.paged_attention_decode(src["q"], k, v, src["tables"], src["lens"], w.scale, w.block_size,
                                       out=out, workspace=ws, stream=st)
        else:
            pkv.paged_attention_decode_shared_prefix(src["q"], k, v, src["tables"], src["lens"], src["gs"],
                                                     src["pl"], w.scale, w.block_size, grouped["max_group"],
                                                     out=out, workspace=ws, stream=st)

    def staged(st):
        dev_buf.copy_(host_buf, non_blocking=True)
        step_calls(st, dbuf, out_d)
        out_h.copy_(out_d, non_blocking=True)

    def direct(st):
        step_calls(st, hbuf, out_h)

    def timed(body):
        stream = torch.cuda.current_stream()
        for _ in range(max(args.warmup, 3)):
            body(stream)
            stream.synchronize()
        # the step as a CUDA graph, recorded once through the same API calls and replayed every
        # step (what a serving loop does with a fixed-shape decode step); eager calls if capture fails
        graph, how = None, "eager API calls"
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body(torch.cuda.current_stream())
            torch.cuda.synchronize()
            graph, how = g, "CUDA graph of the API calls, replayed"
        except Exception as e:  # noqa: BLE001 - any capture failure falls back to the eager step
            how = f"eager API calls (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()

        def step():
            if graph is not None:
                graph.replay()
            else:
                body(stream)
            stream.synchronize()

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        return (time.perf_counter() - t0) / args.steps * 1e3, how

    staged_ms, how = timed(staged)
    res = {"e2e_staged_ms": staged_ms, "h2d": h2d, "d2h": d2h}
    if grouped is None:
        direct_ms, how_d = timed(direct)
        res.update(e2e_step_ms=direct_ms, launch=how_d + "; the kernels read the inputs from page-locked "
                   "host memory over NVLink-C2C and write the output there (no staging copies)")
    else:
        res.update(e2e_step_ms=staged_ms, launch=how + "; one staging copy each way")
    return res


def prepare_cpu_sample(w, seqs, slots, seed):
    """Host inputs of the oracle for sequences `seqs` of the step (generated once, untimed)."""
    from paged_kv_cache_73_gb300 import workloads as wl

    S, H, D, B = w.num_seqs, w.num_heads, w.head_dim, w.block_size
    kc, vc, tabs, lens = w.compact_pools(seqs)
    key, value = wl.new_tokens(S, H, D, seed, "cpu")
    # the new tokens' slots re-expressed in the compact pool's block numbering
    ids = sorted({int(x) for x in w.block_tables[seqs].ravel() if x >= 0})
    remap = {b: i for i, b in enumerate(ids)}
    local = [remap[int(slots[s]) // B] * B + int(slots[s]) % B for s in seqs]
    return {"k": kc.numpy(), "v": vc.numpy(), "tables": tabs, "lens": lens, "slots": local,
            "key": key.numpy()[seqs], "value": value.numpy()[seqs], "q": w.q("cpu").numpy()[seqs],
            "scale": w.scale, "kv_bytes": int(lens.astype(np.int64).sum()) * H * D * 2 * 2}


def cpu_sample_seconds(x):
    """Oracle (fp64, host) over a prepared sample: the new-token writes, then attention."""
    from oracle import attention as oracle_attention
    from oracle import cache_ops as oracle_cache_ops

    t0 = time.perf_counter()
    oracle_cache_ops.reshape_and_cache(x["key"], x["value"], x["k"], x["v"], x["slots"])
    oracle_attention.paged_decode_attention(x["q"], x["k"], x["v"], x["tables"], x["lens"], x["scale"])
    return time.perf_counter() - t0


def _cpu_worker(job):
    """One process of the all-cores CPU baseline: regenerate this worker's share of the sample,
    wait for the others, time the oracle on it."""
    seqs, workload, capacity_seqs, capacity_block, start = job
    x0 = build_step_inputs(SEED, workload, capacity_seqs, capacity_block)
    x = prepare_cpu_sample(x0["w"], seqs, x0["slots"], SEED)
    start.wait()
    t0 = time.time()
    cpu_sample_seconds(x)
    return t0, time.time(), x["kv_bytes"]


def run_cpu_baseline_all_cores(args, seqs):
    """The same sample over every host core: one single-threaded process per core (spawned, before
    any GPU work), the sequences dealt round-robin by length; wall time from the first start to
    the last finish."""
    import multiprocessing as mp
    n = max(1, min(os.cpu_count() or 1, len(seqs)))
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        start = mgr.Barrier(n)
        jobs = [(seqs[i::n], args.workload, args.capacity_seqs, args.capacity_block, start) for i in range(n)]
        with ctx.Pool(n) as pool:
            res = pool.map(_cpu_worker, jobs)
    wall = max(r[1] for r in res) - min(r[0] for r in res)
    kv = sum(r[2] for r in res)
    return {"value": kv / wall / 1e9, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"the same {len(seqs)} sequences over {n} single-threaded processes, {wall:.2f} s"}


def run_cpu_baseline(args, budget_s: float = 12.0):
    x0 = build_step_inputs(SEED, args.workload, args.capacity_seqs, args.capacity_block)
    w, slots = x0["w"], x0["slots"]
    S = w.num_seqs
    order = [int(x) for x in np.argsort(w.context_lens)[::-1]]
    seqs = []
    for a, b in zip(order, order[::-1]):               # alternate long and short sequences
        for s in (a, b):
            if s not in seqs:
                seqs.append(s)
    probe = cpu_sample_seconds(prepare_cpu_sample(w, seqs[:2], slots, SEED))
    n = max(2, min(S, int(budget_s / max(probe / 2, 1e-3))))
    x = prepare_cpu_sample(w, seqs[:n], slots, SEED)
    secs = cpu_sample_seconds(x)
    out = {"value": x["kv_bytes"] / secs / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{n} of the {S} sequences (all {w.num_heads} heads, {int(x['lens'].sum())} tokens), "
                     f"new-token writes + fp64 attention, numpy single-threaded, {secs:.1f} s"}
    if (os.cpu_count() or 1) > 1:
        out["all_cores"] = run_cpu_baseline_all_cores(args, seqs[:n])
    return out


def reduce_over_ranks(maxed, summed, world, device):
    """Max over ranks of `maxed` (times), sum over ranks of `summed` (bytes)."""
    import torch
    t = torch.tensor(list(maxed), dtype=torch.float64, device=device)
    b = torch.tensor(list(summed), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], [float(x) for x in b.tolist()]


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def l2_cache_bytes(dev) -> int:
    import torch
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0) or 132 * 1024 * 1024)


def config_block(args, desc, num_seqs, extra=None, flushed=False):
    c = {"workload": desc, "num_seqs": num_seqs, "num_heads": 40, "head_dim": 128,
         "block_size": args.capacity_block if args.workload == "capacity" else 16,
         "seed": f"{SEED} (+7919*rank)", "kv_storage": "f16",
         "l2": ("L2 flushed before every step (a write of twice the L2 size, outside the timed region); "
                "each step timed by its own events") if flushed
               else "inputs larger than L2: the step reads more than twice the L2 size of distinct K/V"}
    if extra:
        c.update(extra)
    return c


def run_reference(args, rank):
    """The oracle, as it stands, on the host cores: each step one sequence of the workload."""
    if rank != 0:
        return None
    x0 = build_step_inputs(SEED, args.workload, args.capacity_seqs, args.capacity_block)
    w, slots = x0["w"], x0["slots"]
    order = [int(x) for x in np.random.default_rng(0).permutation(w.num_seqs)][:8]
    samples = [prepare_cpu_sample(w, [s], slots, SEED) for s in order]   # generated once, untimed
    for i in range(args.warmup):
        cpu_sample_seconds(samples[i % len(samples)])
    secs, kv = 0.0, 0
    for i in range(args.steps):
        x = samples[i % len(samples)]
        secs += cpu_sample_seconds(x)
        kv += x["kv_bytes"]
    value = kv / secs / 1e9
    sample = f"one sequence (all {w.num_heads} heads) per step, cycling over {len(samples)} of the {w.num_seqs}"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-based generator)",
            "config": config_block(args, x0["desc"], w.num_seqs, {"reference_sample": sample}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample + "; new-token write + fp64 attention"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def headline_line(args, r, world, cpu, step_ms, e2e_ms, attn_ms, staged_ms, attn_med, kv_total, phys_total):
    """The JSON line of a decode run: `r` is this rank's run_gpu result, the times (ms) are maxima
    over ranks and the byte counts sums over ranks."""
    peak, peak_src = measured_hbm_peak()
    achieved = r["attn_bytes"] / (attn_ms * 1e-3) / 1e9
    traffic = None if args.grouped else NCU_TRAFFIC.get(
        (args.workload + ("+append" if r["fused"] else ""), attention_source_sha()))
    value = kv_total / (step_ms * 1e-3) / 1e9
    S = r["num_seqs"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded counter-based generator)",
        "config": config_block(args, r["desc"], S,
                               {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                "partition_tokens": r["part_tokens"], "cow_pairs_per_step": r["n_pairs"],
                                "pool_blocks": r["num_blocks"]}, flushed=r["l2_flushed"]),
        "hbm_frac_of_measured": value / peak,
        "hbm_frac_of_nominal": value / NOMINAL_HBM_GBS,
        "physical_kv_GBps": phys_total / (step_ms * 1e-3) / 1e9,
        "tokens_per_s": S * world / (step_ms * 1e-3),
        "tokens_per_s_40_layer_attention_only": S * world / (40 * step_ms * 1e-3),
        "host_slot_assignment_us": r["host_slot_us"],
        "roofline": {"bound": "hbm",
                     "kernel": ("paged attention call with the new tokens' K/V append (partition + merge "
                                "kernels); bytes include the appended rows read and written"
                                if r["fused"] else "paged attention call (partition + merge kernels)")
                     if r["grouped"] is None
                     else "shared-prefix attention call (prefix partials on tensor cores + partition + merge); "
                          "bytes = distinct K/V slots + q + out",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": r["attn_bytes"],
                     "launch_ms": attn_ms, "launch_ms_median": attn_med,
                     "timed_launches": args.steps if r["l2_flushed"] else (args.steps + EVENT_EVERY - 1) // EVENT_EVERY,
                     "peak_source": peak_src + ", of measured"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if r["copy"] is not None:
        line["copy_blocks_setup"] = r["copy"]
    if r.get("bm") is not None:
        line["block_manager"] = r["bm"]
    if r["grouped"] is not None:
        line["grouped"] = r["grouped"]
    if "e2e_step_ms" in r:
        line["e2e"] = {"value": kv_total / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                       "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                       "ms_per_step": e2e_ms, "launch": r.get("launch", "eager API calls"),
                       "staged_value": kv_total / (staged_ms * 1e-3) / 1e9,
                       "staged_ms_per_step": staged_ms}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}), flush=True)
        sys.exit(1)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    if args.workload in AUX_WORKLOADS:
        from paged_kv_cache_73_gb300 import binding as pkv
        pkv.load()
        line = {"swap": run_swap, "layers40": run_layers40, "prefill": run_prefill}[args.workload](args, dev)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args)                      # before any timing: the oracle runs alone

    from paged_kv_cache_73_gb300 import binding as pkv
    pkv.load()
    r = run_gpu(args, rank, world, dev)

    # whole-job numbers: bytes of all ranks over the slowest rank's time
    (step_ms, e2e_ms, attn_ms, staged_ms, attn_med), (kv_total, phys_total) = reduce_over_ranks(
        [r["step_ms"], r.get("e2e_step_ms", 0.0), r["attn_ms"], r.get("e2e_staged_ms", 0.0), r["attn_ms_median"]],
        [float(r["kv_bytes"]), float(r["phys_bytes"])],
        world, dev)

    if rank == 0:
        line = headline_line(args, r, world, cpu, step_ms, e2e_ms, attn_ms, staged_ms, attn_med, kv_total,
                             phys_total)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
