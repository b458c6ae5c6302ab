"""Decode-step benchmark of the paged K/V-cache path on GB300.

One step = one decode step of the OPT-13B-shaped single-layer batch (64
sequences, 40 heads x 128, block size 16, context lengths ~ U[128, 2048],
physical blocks shuffled): copy_blocks of the step's copy-on-write pairs (none
in this batch), then the 64 new tokens' K/V write and paged decode attention in
one launch (pkv_paged_attention_decode_append).  Batches whose K/V is mostly
shared blocks (served from L2) take reshape_and_cache, then
pkv_paged_attention_decode instead (--step picks either form).  The tables and slots come from the host
block manager.

Prints ONE JSON line (rank 0):
* value: effective KV GB/s, the K/V bytes attention reads per step (logical, a
  shared block counted per reader) over the device time of exactly K steps
  (CUDA events before and after them, nothing in between);
* roofline: the attention call alone, max(200, K) launches back to back after
  the timed region, against the measured HBM copy bandwidth; its median comes
  from a separate loop with events around every launch;
* sustained: at least one second of back-to-back steps, with its own clock
  samples; `clocks` spans the timed region and this segment;
* e2e: a real decode loop through the C ABI from the host.  Every step the
  host block manager assigns the new tokens' slots and builds the tables
  (pkv_bm_append_slots, pkv_bm_block_tables) into page-locked host memory, the
  kernels read them (and q and the new K/V rows) across NVLink-C2C and write
  the output there, and the host waits for it; the contexts grow by one token
  a step.  `graph_replay` is the same step's fixed inputs replayed as a CUDA
  graph;
* configs: the tiny batch, parallel sampling with copy-on-write, the shared
  prefix and the capacity sweep at 1 and 64 sequences: GB/s, the fraction of
  the measured peak and the max abs error of sampled sequences against the
  oracle (whose outputs the CPU-baseline leg computes);
* cpu_baseline: the oracle (numpy fp64) on the whole batch, one host core, and
  one single-threaded process per core.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload opt13b|tiny|parallel_sampling|parallel_sampling_cow|shared_prefix|capacity
                              |beam_search|swap|layers40|prefill]
                  [--capacity-seqs S] [--capacity-block B] [--pool-frac F] [--grouped]
                  [--step auto|fused|unfused]

`--workload swap`, `--workload layers40` and `--workload prefill` print their
own lines (swap_blocks between HBM and page-locked host memory; 40-layer
copy_blocks and reshape_and_cache in one launch; prefill attention over a
cached prefix on the tensor cores) with their own metric names.

--grouped makes the attention call pkv_paged_attention_decode_shared_prefix:
consecutive sequences whose leading blocks are the same physical blocks form a
group whose shared prefix is read once (groups under 8 members still read it
per sequence); the metric is unchanged and `roofline` then counts distinct K/V
slots.

--impl reference times the CPU oracle on the host cores instead: each step the
new-token writes and fp64 attention over the whole batch, whose tables and
slots the oracle's own block manager builds (libpkv.so is not loaded).
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
            "+ the K/V write of 64 new tokens (in the attention launch)")
# seed of each workload's length draws and physical-block permutation: 1000 + its index
WORKLOAD_SEEDS = {"tiny": 1001, "opt13b": 1002, "parallel_sampling": 1003, "parallel_sampling_cow": 1003,
                  "shared_prefix": 1004, "capacity": 1005, "beam_search": 1006}
SEED = WORKLOAD_SEEDS["opt13b"]
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0                                # GB300 HBM3e, nominal
# a step whose distinct K/V is under twice this is preceded by a write of twice the device's L2
L2_NOMINAL_BYTES = 129 * 10 ** 6
ROOFLINE_LAUNCHES = 200                                 # attention calls timed for the roofline, at least
SUSTAINED_S = 1.0                                       # seconds of back-to-back steps, at least
CONFIG_STEPS = 50                                       # timed steps of each entry of `configs`
REF_MAX_KV_BYTES = 2.5e9                                # the oracle arm samples batches larger than this
REF_WALL_S = 150.0                                      # the oracle arm's whole run (warm-up included), about

# dram__bytes_read.sum + dram__bytes_write.sum of one paged-attention call from an ncu capture,
# keyed by (workload, sha256 of the attention source it was taken on); a changed kernel reports
# null until it is captured again.
NCU_TRAFFIC = {
    # the headline step's fused call: partition kernel 1,373,096,704 B read + 4,926,208 B written
    # (the appended rows included), merge kernel 1,280,384 B read (means of two launches each)
    ("opt13b+append", "39ce661f5a57a33b74881bb7a29140e0350bb767558bf3a41d17c172630552dc"): 1_379_303_296,
}

WORKLOADS = ("opt13b", "tiny", "parallel_sampling", "parallel_sampling_cow", "shared_prefix", "capacity",
             "beam_search")
AUX_WORKLOADS = ("swap", "layers40", "prefill")


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer loops (profiling runs)")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' entries (profiling runs)")
    ap.add_argument("--no-sustained", action="store_true", help="skip the roofline and sustained loops (profiling runs)")
    ap.add_argument("--step", choices=["auto", "fused", "unfused"], default="auto",
                    help="fused: the new tokens' K/V write inside the attention launch "
                         "(pkv_paged_attention_decode_append); unfused: reshape_and_cache, then attention; "
                         "auto (default): fused unless shared blocks make up most of the batch's K/V")
    ap.add_argument("--unfused", action="store_true", help="the same as --step unfused")
    ap.add_argument("--grouped", action="store_true",
                    help="read each shared prefix once per group of sequences (shared-prefix decode entry); "
                         "groups come from the block manager's shared leading blocks")
    ap.add_argument("--workload", choices=WORKLOADS + AUX_WORKLOADS, default="opt13b",
                    help="opt13b (the headline batch) or another decode batch of the same shape family")
    ap.add_argument("--capacity-seqs", type=int, default=64, help="capacity workload: sequences (ctx 2048 each)")
    ap.add_argument("--capacity-block", type=int, default=16, help="capacity workload: block size")
    ap.add_argument("--pool-frac", type=float, default=0.0,
                    help="capacity workload: size the pool to this fraction of free HBM (0 = just enough)")
    return ap.parse_args(argv)


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


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured bf16 dense burst (MEASURED_PEAKS.json bf16_tflops; fp16 has the same nominal rate), of measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback 1.9 PFLOP/s bf16 burst"


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

def workload_seed(workload: str) -> int:
    return WORKLOAD_SEEDS.get(workload, SEED)


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


class OracleManager:
    """The oracle's block manager behind the methods of the binding's BlockManager that the bench
    calls, with the same arguments and return shapes.  The reference arm and the CPU-baseline leg
    build their batches with it, so neither loads libpkv.so; a CPU test checks that both managers
    give the bench's batches identical tables, slots and copies."""

    def __init__(self, num_blocks: int, block_size: int, free_order):
        from oracle import block_manager as obm
        self.m = obm.BlockManager(num_blocks, block_size, [int(b) for b in free_order])
        self.num_blocks = num_blocks
        self.block_size = block_size

    @staticmethod
    def _pairs(copies):
        return np.array(copies, dtype=np.int64).reshape(-1, 2)

    def add_seq(self, seq_id, prompt_len):
        return np.array(self.m.add_seq(int(seq_id), int(prompt_len)), dtype=np.int64)

    def fork(self, parent, child):
        self.m.fork(int(parent), int(child))

    def register_prefix(self, prefix_id, length):
        return np.array(self.m.register_prefix(int(prefix_id), int(length)), dtype=np.int64)

    def add_seq_with_prefix(self, seq_id, prefix_id, suffix_len=0):
        slots, copies = self.m.add_seq_with_prefix(int(seq_id), int(prefix_id), int(suffix_len))
        return np.array(slots, dtype=np.int64), self._pairs(copies)

    def extend(self, seq_id, n):
        slots, copies = self.m.extend(int(seq_id), int(n))
        return np.array(slots, dtype=np.int64), self._pairs(copies)

    def append_slots(self, seq_ids):
        slots, copies = [], []
        for s in seq_ids:
            slot, src, dst = self.m.append_slot(int(s))
            slots.append(slot)
            if src >= 0:
                copies.append((src, dst))
        return np.array(slots, dtype=np.int64), self._pairs(copies)

    def block_table(self, seq_id):
        return self.m.block_table(int(seq_id))

    def block_tables(self, seq_ids, max_blocks):
        tables = np.full((len(seq_ids), max_blocks), -1, dtype=np.int32)
        lens = np.zeros(len(seq_ids), dtype=np.int32)
        for i, s in enumerate(seq_ids):
            ids, ctx = self.m.block_table(int(s))
            if len(ids) > max_blocks:
                raise ValueError(f"sequence {s} has {len(ids)} blocks > {max_blocks}")
            tables[i, :len(ids)] = ids
            lens[i] = ctx
        return tables, lens

    def beam_step(self, parents, children, retire):
        res = self.m.beam_step([int(p) for p in parents], [int(c) for c in children], [int(r) for r in retire])
        return (np.array([r[0] for r in res], dtype=np.int64),
                self._pairs([(r[1], r[2]) for r in res if r[1] >= 0]))

    def stats(self):
        return self.m.num_free(), self.m.tail_waste_tokens(), self.m.cow_copies

    def ref_histogram(self, cap=8):
        return np.array(self.m.ref_histogram(cap), dtype=np.int64)

    def counters(self):
        return self.m.counters()


def make_manager(kind: str, num_blocks: int, block_size: int, free_order):
    """The C++ block manager (the product) or, for the oracle's legs, the oracle's."""
    if kind == "oracle":
        return OracleManager(num_blocks, block_size, free_order)
    from paged_kv_cache_73_gb300 import binding as pkv
    return pkv.BlockManager(num_blocks, block_size, free_order)


def block_manager_summary(bm) -> dict:
    """The manager's state after the step's slot assignment: occupancy, sharing and events."""
    free, waste, _ = bm.stats()
    return {"free_blocks": int(free), "tail_waste_tokens": int(waste),
            "ref_histogram": [int(x) for x in bm.ref_histogram(8)], **bm.counters()}


def build_step_inputs(seed: int, workload: str = "opt13b", capacity_seqs: int = 64, capacity_block: int = 16,
                      pool_blocks=None, manager: str = "native"):
    """A decode step's batch built through a host block manager over the recipe's lengths.

    Every sequence is grown to ctx - 1 tokens (a prompt, forked samples whose own tokens are
    placed in one call each, or requests on a registered prefix whose own tokens are placed in the
    same call; copy-on-write where a shared partly filled block is written), then one append per
    sequence gives this step's new-token slots and copy pairs.  `manager` is "native" (the C++
    manager of libpkv.so) or "oracle" (oracle/block_manager.py).
    Returns a dict: w (DecodeWorkload over the manager's tables), slots, pairs (this step's
    copies), setup_pairs (copies made while growing), host_us, desc, manager (the live manager,
    for further steps), seqs, bm (a summary).
    """
    from paged_kv_cache_73_gb300 import workloads as wl

    if workload == "beam_search":
        return build_beam_step(seed, manager=manager)
    if workload == "opt13b":
        recipe = wl.opt13b(seed=seed)
    elif workload == "tiny":
        recipe = wl.tiny(seed=seed)
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
    bm = make_manager(manager, N, B, wl.free_list_order(N, seed))
    seqs = list(range(S))
    setup = []
    if workload.startswith("parallel_sampling"):
        n, prompt = 4, 512 if workload == "parallel_sampling" else 511
        for base in range(0, S, n):
            bm.add_seq(base, prompt)
            for i in range(1, n):
                bm.fork(base, base + i)
        for s in seqs:                                   # each sample's own tokens, in one call
            _, pr = bm.extend(s, int(lens[s]) - 1 - prompt)
            setup += pr.tolist()
    elif workload == "shared_prefix":
        prefix = 1024
        bm.register_prefix(0, prefix)
        for s in seqs:                                   # the request and its own tokens, in one call
            _, pr = bm.add_seq_with_prefix(s, 0, int(lens[s]) - 1 - prefix)
            setup += pr.tolist()
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
    elif workload == "tiny":
        desc = f"tiny: 3 seqs, ctx 7/5/12, 2 heads x 64, block 4, {N} pool blocks, shuffled"
    else:
        desc = f"{workload}: {recipe.notes}, 40 x 128, block {B}, shuffled blocks"
    return {"w": w, "slots": slots, "pairs": pairs, "setup_pairs": np.array(setup, dtype=np.int64).reshape(-1, 2),
            "host_us": host_us, "desc": desc, "workload": workload, "manager": bm, "seqs": seqs,
            "bm": block_manager_summary(bm)}


def build_beam_step(seed: int, requests: int = 16, width: int = 4, beam_steps: int = 128, B: int = 16,
                    manager: str = "native"):
    """Beam search through the block manager: each request keeps `width` candidates; every step
    each new candidate picks a parent among the current ones (seeded), the old beam is retired and
    shared partly filled blocks are copied once per extra sibling.  The measured step is one more
    beam step: its copies, its new tokens' writes and attention over all candidates."""
    from paged_kv_cache_73_gb300 import workloads as wl

    H, D = 40, 128
    rng = np.random.default_rng(seed)
    prompts = rng.integers(256, 1025, size=requests)
    N = int(2 * (sum(-(-int(p) // B) for p in prompts) + requests * width * (beam_steps // B + 3)))
    bm = make_manager(manager, N, B, wl.free_list_order(N, seed))
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
            "workload": "beam_search", "manager": bm, "seqs": seqs, "bm": block_manager_summary(bm)}


# The fused step (the new rows' write inside the attention launch) is 1 % faster on the OPT-13B-shaped
# batch, whose K/V streams from HBM, but 2-3.5 % slower where L2 serves shared blocks (parallel
# sampling 140.0 against 137.7 us, 256 shared-prefix requests 531 against 513): there the
# partitions are short and the appending CTA's extra work shows.  The host knows which case it has
# from the block manager's sharing: distinct K/V well below the logical K/V.
FUSED_MIN_DISTINCT = 0.75


def use_fused(args, w) -> bool:
    """The step form for batch w: --step fused / unfused, or by the batch's sharing (auto)."""
    step = "unfused" if args.unfused else args.step
    if step != "auto":
        return step == "fused"
    return w.physical_kv_bytes() >= FUSED_MIN_DISTINCT * w.logical_kv_bytes()


def needs_flush(w) -> bool:
    """A step whose distinct K/V would stay in L2 between steps is preceded by an L2 flush."""
    return w.physical_kv_bytes() < 2 * L2_NOMINAL_BYTES


# ---- the GPU arm -----------------------------------------------------------------------------------

class Step:
    """One decode step of a batch on the device: pools, inputs and the calls, through the binding."""

    def __init__(self, x, dev, fused=True, grouped=False):
        import torch
        from paged_kv_cache_73_gb300 import binding as pkv
        from paged_kv_cache_73_gb300 import workloads as wl
        self.pkv = pkv
        self.x = x
        w = self.w = x["w"]
        S, H, D, B, MB = w.num_seqs, w.num_heads, w.head_dim, w.block_size, w.max_blocks_per_seq
        self.k, self.v = w.pools(dev)
        self.q = w.q(dev)
        self.key, self.value = wl.new_tokens(S, H, D, w.seed, dev)
        self.tables = torch.from_numpy(w.block_tables).to(dev)
        self.lens = torch.from_numpy(w.context_lens).to(dev)
        self.slots = torch.from_numpy(np.ascontiguousarray(x["slots"])).to(dev)
        self.pairs = torch.from_numpy(np.ascontiguousarray(x["pairs"])).to(dev)
        self.n_pairs = int(x["pairs"].shape[0])
        self.out = torch.empty_like(self.q)
        self.ws = pkv.workspace_for(S, H, D, MB, B, dev)
        self.part_tokens, self.attn_kernels = pkv.paged_attention_plan(S, H, D, MB, B)
        self.stream = torch.cuda.current_stream()
        self.grouped = None
        if grouped:
            gs_h, pl_h = shared_prefix_groups(w.block_tables, w.context_lens, B)
            n_ws = pkv.paged_attention_shared_prefix_workspace_size(S, H, D, MB, B)
            self.grouped = {"gs": torch.from_numpy(gs_h).to(dev), "pl": torch.from_numpy(pl_h).to(dev),
                            "max_group": int(np.max(np.diff(gs_h))), "groups": int(len(pl_h)),
                            "prefix_tokens": int(pl_h.sum()), "gs_h": gs_h, "pl_h": pl_h}
            self.ws = torch.empty(max(n_ws, 16), dtype=torch.uint8, device=dev)
            self.attn_kernels = 3                        # prefix partials, partitions, merge
        self.fused = fused and not grouped
        self.kernels_per_step = (1 if self.n_pairs else 0) + (0 if self.fused else 1) + self.attn_kernels

    def attention(self):
        """The step's attention call (with the new rows' write when fused)."""
        pkv, w, st = self.pkv, self.w, self.stream
        if self.fused:
            pkv.paged_attention_decode_append(self.q, self.key, self.value, self.slots, self.k, self.v, self.tables,
                                              self.lens, w.scale, w.block_size, out=self.out, workspace=self.ws,
                                              stream=st)
        elif self.grouped is None:
            pkv.paged_attention_decode(self.q, self.k, self.v, self.tables, self.lens, w.scale, w.block_size,
                                       out=self.out, workspace=self.ws, stream=st)
        else:
            g = self.grouped
            pkv.paged_attention_decode_shared_prefix(self.q, self.k, self.v, self.tables, self.lens, g["gs"], g["pl"],
                                                     w.scale, w.block_size, g["max_group"], out=self.out,
                                                     workspace=self.ws, stream=st)

    def __call__(self):
        pkv, st = self.pkv, self.stream
        if self.n_pairs:
            pkv.copy_blocks([self.k], [self.v], self.pairs, stream=st)
        if not self.fused:
            pkv.reshape_and_cache(self.key, self.value, self.k, self.v, self.slots, stream=st)
        self.attention()

    def attention_bytes(self) -> int:
        """Algorithmic bytes of the attention call: K/V rows, q, out, tables and lengths; plus the
        new rows read and written when fused; the distinct K/V slots when grouped."""
        w = self.w
        if self.grouped is not None:
            return w.physical_kv_bytes() + w.num_seqs * w.num_heads * w.head_dim * 2 * 2
        extra = 4 * w.num_seqs * w.num_heads * w.head_dim * 2 if self.fused else 0
        return attention_algorithmic_bytes(w) + extra


def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_steps(fn, n, stream, flush_buf=None):
    """Device time (ms) of n calls of fn: with flush_buf, each call follows a write of the buffer
    and has its own events (returns the per-call times); else one event pair around all n (returns
    [mean])."""
    import torch
    if flush_buf is None:
        a, b = _events(2)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) / n]
    evs = [_events(2) for _ in range(n)]
    for i in range(n):
        flush_buf.fill_(i & 255)
        evs[i][0].record(stream)
        fn()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_each(fn, n, stream, flush_buf=None):
    """Per-call device times (ms) of n calls, each between its own events (and after a flush)."""
    import torch
    evs = [_events(2) for _ in range(n)]
    for i in range(n):
        if flush_buf is not None:
            flush_buf.fill_(i & 255)
        evs[i][0].record(stream)
        fn()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_gpu(args, rank, world, dev, cpu_refs=None):
    import torch

    seed = workload_seed(args.workload) + 7919 * rank  # weak scaling: each rank its own batch
    x = build_step_inputs(seed, args.workload, args.capacity_seqs, args.capacity_block,
                          pool_blocks_for(args, dev))
    st = Step(x, dev, fused=use_fused(args, x["w"]), grouped=args.grouped)
    pkv, w, stream = st.pkv, st.w, st.stream
    H, D, B = w.num_heads, w.head_dim, w.block_size

    copy = None
    if len(x["setup_pairs"]):
        # the copy-on-write copies made while the batch grew, as one copy_blocks call
        sp = torch.from_numpy(np.ascontiguousarray(x["setup_pairs"])).to(dev)
        fn = lambda: pkv.copy_blocks([st.k], [st.v], sp, stream=stream)       # noqa: E731
        for _ in range(5):
            fn()
        ms = time_steps(fn, 20, stream)[0]
        moved = 2 * 2 * len(sp) * H * B * D * 2           # K and V, read and written
        copy = {"pairs": int(len(sp)), "ms": ms, "GB/s": moved / (ms * 1e-3) / 1e9}

    # clocks sampled from before the warm-up on; stopped at exit as well, should the run raise
    clocks = ClockSampler(physical_gpu_index(torch.cuda.current_device())).start()
    atexit.register(clocks.stop)
    for _ in range(max(args.warmup, 3)):
        st()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0

    K = args.steps
    flush = needs_flush(w)
    scratch = torch.empty(2 * l2_cache_bytes(dev), dtype=torch.uint8, device=dev) if flush else None
    barrier(world)
    torch.cuda.synchronize()
    # the timed region: exactly K steps, nothing between them (or, for a batch L2 would hold, each
    # step after a write of twice the L2 size and between its own events)
    t0 = time.time()
    times = time_steps(st, K, stream, scratch)
    t1 = time.time()
    barrier(world)
    step_ms = sum(times) / len(times)
    region = (t0, t1)
    code = pkv.device_error()
    assert code == 0, f"device check {code}"

    res = {"step_ms": step_ms, "l2_flushed": flush, "kv_bytes": w.logical_kv_bytes(),
           "phys_bytes": w.physical_kv_bytes(), "attn_bytes": st.attention_bytes(), "fused": st.fused,
           "grouped": None if st.grouped is None
           else {k_: st.grouped[k_] for k_ in ("groups", "max_group", "prefix_tokens")},
           "num_seqs": w.num_seqs, "launches": K * st.kernels_per_step, "kernels_per_step": st.kernels_per_step,
           "part_tokens": st.part_tokens, "host_slot_us": x["host_us"], "n_pairs": st.n_pairs, "copy": copy,
           "desc": x["desc"], "num_blocks": w.num_blocks, "bm": x["bm"]}

    if not args.no_sustained:
        # roofline: the attention call alone, at least ROOFLINE_LAUNCHES launches back to back (each
        # after a flush and between its own events for a batch L2 would hold); the median of a
        # separate loop with events around every launch (an event between two launches stops the
        # next one from overlapping the previous one's tail, so these run a little longer)
        n_launch = max(ROOFLINE_LAUNCHES, K)
        lt = time_steps(st.attention, n_launch, stream, scratch)
        iso = time_each(st.attention, n_launch, stream, scratch)
        res.update(attn_ms=sum(lt) / len(lt), attn_ms_median=statistics.median(iso), timed_launches=n_launch,
                   attn_loop="back to back, one event pair around all launches" if scratch is None
                   else "each launch after an L2 flush, between its own events")
        # sustained: at least SUSTAINED_S seconds of back-to-back steps, with their own clock samples
        n_sus = max(K, int(math.ceil(SUSTAINED_S * 1e3 / max(step_ms, 1e-3))))
        ts0 = time.time()
        sus = time_steps(st, n_sus, stream, scratch)
        ts1 = time.time()
        sus_ms = sum(sus) / len(sus)
        sus_clocks = clocks.summary(ts0, ts1)
        res["sustained"] = {"steps": n_sus, "seconds": ts1 - ts0, "ms_per_step": sus_ms,
                            "kv_bytes": w.logical_kv_bytes() * n_sus, "device_s": sus_ms * n_sus * 1e-3,
                            "clocks": sus_clocks}
        res["clocks"] = clocks.summary(t0, ts1)
        if res["clocks"] is not None:
            res["clocks"]["window"] = ("from the start of the timed region to the end of the sustained segment "
                                       "(the roofline loops and the sustained steps follow the timed steps)")
    else:
        iso = time_each(st.attention, max(3, min(K, 20)), stream, scratch)
        res.update(attn_ms=sum(iso) / len(iso), attn_ms_median=statistics.median(iso), timed_launches=len(iso),
                   attn_loop="events around every launch", clocks=None)
    res["clocks_timed_region"] = clocks.summary(*region)
    if res["clocks"] is None:
        res["clocks"] = res["clocks_timed_region"]
    clocks.stop()
    assert pkv.device_error() == 0

    if not args.no_e2e:
        res["e2e_loop"] = run_e2e_loop(args, st, dev)
        res["e2e_replay"] = run_e2e_replay(args, st, dev)
    del scratch
    if rank == 0 and not args.no_configs:
        res["configs"] = run_configs(args, dev, cpu_refs)
    return res


def run_e2e_loop(args, st, dev):
    """A decode loop through the C ABI, timed on the host clock.  Each step the C++ block manager
    assigns the new tokens' slots (pkv_bm_append_slots) and writes the padded tables
    (pkv_bm_block_tables) into page-locked host buffers; the kernels read those, q and the new K/V
    rows across NVLink-C2C and write the output into page-locked host memory; the host waits for
    the output.  The contexts grow by one token a step.

    A step's slot assignment needs no result of the step before, so the host assigns step i+1's
    slots and tables into the second of two buffer sets while the kernels of step i run, as a
    serving loop would.  The direct form calls the C entry points with the buffers' addresses, as
    a C caller does.  With --grouped the step's inputs are copied to the device in one packed copy
    and the output back (that entry loads q by TMA from device memory), through the binding."""
    import ctypes
    import torch
    pkv, w, x = st.pkv, st.w, st.x
    bm, seqs = x["manager"], x["seqs"]
    S, H, D, B, N = w.num_seqs, w.num_heads, w.head_dim, w.block_size, w.num_blocks
    warm = max(args.warmup, 3)
    free = int(bm.stats()[0])
    # steps the free blocks carry: each sequence opens a block at most once every B tokens (and
    # copies at most one block on its first append)
    cap = (free // max(S, 1) - 2) * B
    n = min(args.steps, cap - warm - 1)
    if n < 1:
        return {"skipped": f"the pool's {free} free blocks carry no {warm} + 1 steps"}
    max_blocks = w.max_blocks_per_seq + -(-(warm + n + 2) // B) + 1
    staged = st.grouped is not None
    if staged:
        n_ws = pkv.paged_attention_shared_prefix_workspace_size(S, H, D, max_blocks, B)
        ws = torch.empty(max(n_ws, 16), dtype=torch.uint8, device=dev)
    else:
        ws = pkv.workspace_for(S, H, D, max_blocks, B, dev)
    pin = lambda t: t.cpu().contiguous().pin_memory()                        # noqa: E731
    q_h, key_h, value_h = pin(st.q), pin(st.key), pin(st.value)
    out_h = torch.empty(tuple(st.q.shape), dtype=torch.float16).pin_memory()

    class Buf:
        def __init__(self):
            self.slots = torch.zeros(S, dtype=torch.int64).pin_memory()
            self.pairs = torch.zeros((max(S, 1), 2), dtype=torch.int64).pin_memory()
            self.tables = torch.full((S, max_blocks), -1, dtype=torch.int32).pin_memory()
            self.lens = torch.zeros(S, dtype=torch.int32).pin_memory()
            self.npairs = 0
            self.tokens = 0

    bufs = [Buf(), Buf()]
    lib = pkv.load()
    ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
    ncow = ctypes.c_int(0)
    handle = bm._h
    stream = st.stream
    sh = stream.cuda_stream
    kp = (ctypes.c_void_p * 1)(st.k.data_ptr())
    vp = (ctypes.c_void_p * 1)(st.v.data_ptr())
    ws_ptr = None if ws is None else ws.data_ptr()
    ws_bytes = 0 if ws is None else ws.numel()
    host_s = [0.0]

    def check(rc):
        if rc != 0:
            raise pkv.PkvError(rc, lib.pkv_last_error().decode(errors="replace"))

    def prep(b):
        """The host's part of a step: slots, copies, tables and lengths into buffer set b."""
        h0 = time.perf_counter()
        check(lib.pkv_bm_append_slots(handle, ids.ctypes.data, S, b.slots.data_ptr(), b.pairs.data_ptr(),
                                      ctypes.byref(ncow)))
        b.npairs = ncow.value
        check(lib.pkv_bm_block_tables(handle, ids.ctypes.data, S, b.tables.data_ptr(), max_blocks, b.lens.data_ptr()))
        b.tokens = int(b.lens.numpy().sum(dtype=np.int64))
        host_s[0] += time.perf_counter() - h0

    if staged:
        dev_in = {n_: torch.empty_like(t, device=dev) for n_, t in
                  (("slots", bufs[0].slots), ("pairs", bufs[0].pairs), ("tables", bufs[0].tables),
                   ("lens", bufs[0].lens))}
        out_d = torch.empty_like(st.q)

    def launch(b, sh_=None):
        """The device part of a step, enqueued on the stream."""
        sh_ = sh if sh_ is None else sh_
        if not staged:
            if b.npairs:
                check(lib.pkv_copy_blocks(kp, vp, 1, b.pairs.data_ptr(), b.npairs, H, D, B, N, sh_))
            if st.fused:
                check(lib.pkv_paged_attention_decode_append(
                    q_h.data_ptr(), key_h.data_ptr(), value_h.data_ptr(), b.slots.data_ptr(), st.k.data_ptr(),
                    st.v.data_ptr(), b.tables.data_ptr(), b.lens.data_ptr(), S, H, D, N, max_blocks, w.scale, B,
                    out_h.data_ptr(), ws_ptr, ws_bytes, sh_))
            else:
                check(lib.pkv_reshape_and_cache(key_h.data_ptr(), value_h.data_ptr(), st.k.data_ptr(),
                                                st.v.data_ptr(), b.slots.data_ptr(), S, H, D, B, N, sh_))
                check(lib.pkv_paged_attention_decode(
                    q_h.data_ptr(), st.k.data_ptr(), st.v.data_ptr(), b.tables.data_ptr(), b.lens.data_ptr(), S, H,
                    D, N, max_blocks, w.scale, B, out_h.data_ptr(), ws_ptr, ws_bytes, sh_))
            return
        for n_ in ("slots", "tables", "lens"):
            dev_in[n_].copy_(getattr(b, n_), non_blocking=True)
        if b.npairs:
            dev_in["pairs"][:b.npairs].copy_(b.pairs[:b.npairs], non_blocking=True)
            pkv.copy_blocks([st.k], [st.v], dev_in["pairs"][:b.npairs], stream=stream)
        pkv.reshape_and_cache(st.key, st.value, st.k, st.v, dev_in["slots"], stream=stream)
        g = st.grouped
        pkv.paged_attention_decode_shared_prefix(st.q, st.k, st.v, dev_in["tables"], dev_in["lens"], g["gs"], g["pl"],
                                                 w.scale, B, g["max_group"], out=out_d, workspace=ws, stream=stream)
        out_h.copy_(out_d, non_blocking=True)

    # Each buffer set's attention call reads fixed addresses, so it is captured once as a CUDA
    # graph (the same C-ABI calls, recorded) and launched with one call per step; a step's
    # copy-on-write copies, when it has any, run before it as an ordinary call.
    graphs = [None, None]
    how = "eager C-ABI calls"
    if not staged:
        try:
            for k_, b_ in enumerate(bufs):
                b_.npairs = 0
                g_ = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_):
                    cap = torch.cuda.current_stream().cuda_stream
                    launch(b_, cap)
                graphs[k_] = g_
            torch.cuda.synchronize()
            how = "a CUDA graph of each buffer set's attention call (the C-ABI calls, captured once)"
        except Exception as e:  # noqa: BLE001 - any capture failure falls back to eager calls
            graphs = [None, None]
            how = f"eager C-ABI calls (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()

    def run(i, b):
        if graphs[i % 2] is None:
            launch(b)
            return
        if b.npairs:
            check(lib.pkv_copy_blocks(kp, vp, 1, b.pairs.data_ptr(), b.npairs, H, D, B, N, sh))
        graphs[i % 2].replay()

    def loop(steps):
        kv, copies = 0, 0
        prep(bufs[0])
        for i in range(steps):
            b = bufs[i % 2]
            run(i, b)
            if i + 1 < steps:
                prep(bufs[(i + 1) % 2])        # the next step's slots and tables, beside the kernels
            stream.synchronize()               # this step's output is in page-locked host memory
            kv += b.tokens * H * D * 2 * 2
            copies += b.npairs
        return kv, copies

    loop(warm)
    assert pkv.device_error() == 0
    host_s[0] = 0.0
    t0 = time.perf_counter()
    kv, copies = loop(n)
    secs = time.perf_counter() - t0
    assert pkv.device_error() == 0
    b = bufs[0]
    step_in = (q_h.nbytes + key_h.nbytes + value_h.nbytes + b.slots.nbytes + b.tables.nbytes + b.lens.nbytes)
    return {"steps": n, "seconds": secs, "kv_bytes": kv, "ms_per_step": secs / n * 1e3,
            "host_a1_us_per_step": host_s[0] / n * 1e6, "copies": copies,
            "h2d_bytes_per_step": step_in + 16 * copies // max(n, 1), "d2h_bytes_per_step": out_h.nbytes,
            "staged": staged, "launch_form": how}


def run_e2e_replay(args, st, dev):
    """The step's fixed inputs through the C ABI in page-locked host memory, replayed as a CUDA
    graph of the API calls (what a serving loop does with a fixed-shape decode step), two ways:
    direct (the kernels read the inputs and write the output across NVLink-C2C) and staged (one
    packed host->device copy of the inputs and a device->host copy of the output); the host waits
    for the output every step.  A grouped step is staged only (q is loaded by TMA)."""
    import torch
    pkv, w, x = st.pkv, st.w, st.x
    parts = {"q": st.q.cpu(), "key": st.key.cpu(), "value": st.value.cpu(),
             "slots": torch.from_numpy(np.ascontiguousarray(x["slots"])),
             "pairs": torch.from_numpy(np.ascontiguousarray(x["pairs"])),
             "tables": torch.from_numpy(w.block_tables), "lens": torch.from_numpy(w.context_lens)}
    if st.grouped is not None:
        parts["gs"] = torch.from_numpy(st.grouped["gs_h"])
        parts["pl"] = torch.from_numpy(st.grouped["pl_h"])
    # one pinned byte buffer holding every input at a 256-byte-aligned offset, and its device twin
    offs, total = {}, 0
    for n_, t in parts.items():
        offs[n_] = total
        total += -(-(t.numel() * t.element_size()) // 256) * 256
    host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    dbuf, hbuf = {}, {}
    for n_, t in parts.items():
        nbytes = t.numel() * t.element_size()
        host_buf[offs[n_]:offs[n_] + nbytes].copy_(t.contiguous().view(-1).view(torch.uint8))
        dbuf[n_] = dev_buf[offs[n_]:offs[n_] + nbytes].view(t.dtype).view(t.shape)
        hbuf[n_] = host_buf[offs[n_]:offs[n_] + nbytes].view(t.dtype).view(t.shape)
    out_h = torch.empty(tuple(st.q.shape), dtype=torch.float16).pin_memory()
    out_d = torch.empty_like(st.q)
    h2d = sum(t.numel() * t.element_size() for t in parts.values())
    B = w.block_size

    def step_calls(s_, src, out):
        if st.n_pairs:
            pkv.copy_blocks([st.k], [st.v], src["pairs"], stream=s_)
        if st.fused:
            pkv.paged_attention_decode_append(src["q"], src["key"], src["value"], src["slots"], st.k, st.v,
                                              src["tables"], src["lens"], w.scale, B, out=out, workspace=st.ws,
                                              stream=s_)
            return
        pkv.reshape_and_cache(src["key"], src["value"], st.k, st.v, src["slots"], stream=s_)
        if st.grouped is None:
            pkv.paged_attention_decode(src["q"], st.k, st.v, src["tables"], src["lens"], w.scale, B, out=out,
                                       workspace=st.ws, stream=s_)
        else:
            pkv.paged_attention_decode_shared_prefix(src["q"], st.k, st.v, src["tables"], src["lens"], src["gs"],
                                                     src["pl"], w.scale, B, st.grouped["max_group"], out=out,
                                                     workspace=st.ws, stream=s_)

    def staged(s_):
        dev_buf.copy_(host_buf, non_blocking=True)
        step_calls(s_, dbuf, out_d)
        out_h.copy_(out_d, non_blocking=True)

    def direct(s_):
        step_calls(s_, hbuf, out_h)

    def timed(body):
        stream = torch.cuda.current_stream()
        for _ in range(max(args.warmup, 3)):
            body(stream)
            stream.synchronize()
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

        def one():
            if graph is not None:
                graph.replay()
            else:
                body(stream)
            stream.synchronize()

        for _ in range(3):
            one()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            one()
        return (time.perf_counter() - t0) / args.steps * 1e3, how

    staged_ms, how = timed(staged)
    res = {"staged_ms_per_step": staged_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_h.nbytes}
    if st.grouped is None:
        direct_ms, how_d = timed(direct)
        res.update(ms_per_step=direct_ms, launch=how_d + "; the kernels read the fixed inputs from page-locked "
                   "host memory over NVLink-C2C and write the output there (no staging copies)")
    else:
        res.update(ms_per_step=staged_ms, launch=how + "; one staging copy each way")
    return res


# ---- the other configurations ----------------------------------------------------------------------

# (name, workload, capacity sequences)
CONFIG_RUNS = (("tiny", "tiny", 0), ("parallel_sampling_cow", "parallel_sampling_cow", 0),
               ("shared_prefix", "shared_prefix", 0), ("capacity_S1", "capacity", 1),
               ("capacity_S64", "capacity", 64))


def config_sample(w, name):
    """Sequences of a configuration the oracle checks: all of the tiny batch, else the longest and
    the shortest (the first and last when all are equally long)."""
    if name == "tiny":
        return list(range(w.num_seqs))
    lens = w.context_lens
    a, b = int(np.argmax(lens)), int(np.argmin(lens))
    if a == b:
        b = w.num_seqs - 1
    return sorted({a, b})


def run_configs(args, dev, cpu_refs):
    """The other workloads of the path, each as the bench's step on one GPU: effective KV GB/s over
    CONFIG_STEPS steps (L2 flushed before each step where L2 would hold the batch), the fraction of
    the measured HBM peak, and the max abs error of sampled sequences against the oracle outputs
    the CPU-baseline leg computed on the same batch (built there by the oracle's block manager;
    the sampled table rows are compared too), with that leg's oracle time on them (one core).  The parallel-sampling entry also times its 96
    copy-on-write copies as one copy_blocks call and checks them byte for byte."""
    import torch
    peak, _ = measured_hbm_peak()
    out = {}
    for name, workload, cap_seqs in CONFIG_RUNS:
        x = build_step_inputs(workload_seed(workload), workload, cap_seqs or 64, 16)
        st = Step(x, dev, fused=use_fused(args, x["w"]))
        pkv, w = st.pkv, st.w
        flush = needs_flush(w)
        scratch = torch.empty(2 * l2_cache_bytes(dev), dtype=torch.uint8, device=dev) if flush else None
        st()
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        entry = {"workload": x["desc"], "num_seqs": w.num_seqs, "step": "fused" if st.fused else "unfused",
                 "logical_kv_bytes": w.logical_kv_bytes(),
                 "physical_kv_bytes": w.physical_kv_bytes(), "l2_flushed": flush, "steps": CONFIG_STEPS}
        seqs = config_sample(w, name)
        ref = None if cpu_refs is None else cpu_refs.get(name)
        if ref is not None:
            assert ref["seqs"] == seqs
            assert np.array_equal(ref["tables"], w.block_tables[seqs]), "oracle-built tables differ"
            got = st.out[seqs].double().cpu().numpy()
            entry["max_abs_err"] = float(np.max(np.abs(got - ref["out"])))
            entry["checked_seqs"] = seqs
            entry["cpu_oracle"] = {"GB/s": ref["cpu_kv_bytes"] / max(ref["cpu_s"], 1e-9) / 1e9, "cores": 1,
                                   "kind": "oracle",
                                   "sample": f"the {len(seqs)} checked sequences, {ref['cpu_s'] * 1e3:.1f} ms"}
        else:
            entry["max_abs_err"] = None
        for _ in range(3):
            st()
        times = time_steps(st, CONFIG_STEPS, st.stream, scratch)
        ms = sum(times) / len(times)
        entry.update(step_ms=ms, **{"GB/s": w.logical_kv_bytes() / (ms * 1e-3) / 1e9,
                                    "physical_GB/s": w.physical_kv_bytes() / (ms * 1e-3) / 1e9})
        entry["frac_of_measured"] = entry["GB/s"] / peak
        entry["attention_bytes_GB/s"] = st.attention_bytes() / (ms * 1e-3) / 1e9
        if len(x["setup_pairs"]):
            sp = torch.from_numpy(np.ascontiguousarray(x["setup_pairs"])).to(dev)
            fn = lambda: pkv.copy_blocks([st.k], [st.v], sp, stream=st.stream)   # noqa: E731
            fn()
            torch.cuda.synchronize()
            src, dst = sp[:, 0], sp[:, 1]
            exact = bool(torch.equal(st.k[dst].view(torch.int16), st.k[src].view(torch.int16)) and
                         torch.equal(st.v[dst].view(torch.int16), st.v[src].view(torch.int16)))
            cms = time_steps(fn, 20, st.stream)[0]
            moved = 2 * 2 * len(sp) * w.num_heads * w.block_size * w.head_dim * 2
            entry["copy_blocks"] = {"pairs": int(len(sp)), "ms": cms, "GB/s": moved / (cms * 1e-3) / 1e9,
                                    "bit_exact": exact}
        assert pkv.device_error() == 0
        out[name] = entry
        del st, scratch
        torch.cuda.empty_cache()
    return out


# ---- auxiliary workloads ---------------------------------------------------------------------------

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
    gbs = lambda ms: payload / (ms * 1e-3) / 1e9                       # noqa: E731
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
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9                           # noqa: E731
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
    attn = lambda: pkv.paged_attention_prefill(q, k, v, tables, lens, qsd, w.scale, B, maxq, out=out)  # noqa: E731

    def step():
        pkv.reshape_and_cache(key, value, k, v, slots_d)
        attn()

    # long prompts with nothing cached: 8 x 4096 tokens, causal over themselves
    wl2 = wl.custom(SEED + 5, [4096] * 8, H, D, B, name="prefill_8x4096")
    k2, v2 = wl2.pools(dev)
    qs2 = np.arange(0, 8 * 4096 + 1, 4096, dtype=np.int32)
    q2 = wl.dense_tensor((8 * 4096, H, D), SEED + 1, wl.STREAM_Q, dev)
    out2 = torch.empty_like(q2)
    t2, l2, qs2d = (torch.from_numpy(a).to(dev) for a in (wl2.block_tables, wl2.context_lens, qs2))
    flops2 = 8 * 4 * D * H * (4096 * 4097 // 2)
    attn2 = lambda: pkv.paged_attention_prefill(q2, k2, v2, t2, l2, qs2d, wl2.scale, B, 4096, out=out2)  # noqa: E731

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


# ---- the oracle on the host cores -------------------------------------------------------------------

def prepare_cpu_sample(w, seqs, slots, pairs, seed):
    """Host inputs of the oracle for sequences `seqs` of the step (generated once, untimed): the
    blocks their tables map (plus the source of every copy into one of them), regenerated on the
    CPU into a compact pool, and the step's copies and new-token slots renumbered into it."""
    from paged_kv_cache_73_gb300 import workloads as wl

    S, H, D, B = w.num_seqs, w.num_heads, w.head_dim, w.block_size
    seqs = list(seqs)
    mapped = {int(b) for b in w.block_tables[seqs].ravel() if b >= 0}
    copies = [(int(a), int(b)) for a, b in np.asarray(pairs).reshape(-1, 2) if int(b) in mapped]
    kc, vc, tabs, lens, ids = w.compact_pools_with(seqs, [a for a, _ in copies])
    remap = {b: i for i, b in enumerate(ids)}
    key, value = wl.new_tokens(S, H, D, seed, "cpu")
    local = [remap[int(slots[s]) // B] * B + int(slots[s]) % B for s in seqs]
    return {"k": kc.numpy(), "v": vc.numpy(), "tables": tabs, "lens": lens, "slots": local,
            "pairs": [(remap[a], remap[b]) for a, b in copies],
            "key": key.numpy()[seqs], "value": value.numpy()[seqs], "q": w.q("cpu").numpy()[seqs],
            "scale": w.scale, "kv_bytes": int(lens.astype(np.int64).sum()) * H * D * 2 * 2}


def cpu_sample_run(x):
    """The oracle (fp64, host) over a prepared sample: the step's copies, the new-token writes,
    then attention.  Returns (seconds, output)."""
    from oracle import attention as oracle_attention
    from oracle import cache_ops as oracle_cache_ops

    t0 = time.perf_counter()
    if x["pairs"]:
        oracle_cache_ops.copy_blocks([x["k"]], [x["v"]], x["pairs"])
    oracle_cache_ops.reshape_and_cache(x["key"], x["value"], x["k"], x["v"], x["slots"])
    out = oracle_attention.paged_decode_attention(x["q"], x["k"], x["v"], x["tables"], x["lens"], x["scale"])
    return time.perf_counter() - t0, out


def cpu_sample_seconds(x):
    return cpu_sample_run(x)[0]


def _cpu_worker(job):
    """One process of the all-cores CPU baseline: regenerate this worker's share of the sample
    (the batch built by the oracle's block manager), wait for the others, time the oracle on it."""
    seqs, workload, capacity_seqs, capacity_block, start = job
    x0 = build_step_inputs(workload_seed(workload), workload, capacity_seqs, capacity_block, manager="oracle")
    x = prepare_cpu_sample(x0["w"], seqs, x0["slots"], x0["pairs"], workload_seed(workload))
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


def cpu_config_refs():
    """Oracle outputs of the sampled sequences of every entry of `configs` (the batch built by the
    oracle's block manager; the step's copies and new-token writes, then attention)."""
    refs = {}
    for name, workload, cap_seqs in CONFIG_RUNS:
        seed = workload_seed(workload)
        x = build_step_inputs(seed, workload, cap_seqs or 64, 16, manager="oracle")
        w = x["w"]
        seqs = config_sample(w, name)
        sample = prepare_cpu_sample(w, seqs, x["slots"], x["pairs"], seed)
        secs, out = cpu_sample_run(sample)
        refs[name] = {"seqs": seqs, "out": out, "tables": w.block_tables[seqs].copy(), "cpu_s": secs,
                      "cpu_kv_bytes": sample["kv_bytes"]}
    return refs


def run_cpu_baseline(args, budget_s: float = 12.0):
    """The CPU-baseline leg: the oracle as it stands, on the batch its own block manager builds,
    timed on one host core over as many sequences as fit the budget (alternately long and short),
    and on every core; plus the oracle outputs the `configs` entries are checked against."""
    seed = workload_seed(args.workload)
    x0 = build_step_inputs(seed, args.workload, args.capacity_seqs, args.capacity_block, manager="oracle")
    w, slots, pairs = x0["w"], x0["slots"], x0["pairs"]
    S = w.num_seqs
    order = [int(i) for i in np.argsort(w.context_lens)[::-1]]
    seqs = []
    for a, b in zip(order, order[::-1]):               # alternate long and short sequences
        for s in (a, b):
            if s not in seqs:
                seqs.append(s)
    probe = cpu_sample_seconds(prepare_cpu_sample(w, seqs[:2], slots, pairs, seed))
    n = max(2, min(S, int(budget_s / max(probe / 2, 1e-3))))
    x = prepare_cpu_sample(w, seqs[:n], slots, pairs, seed)
    secs = cpu_sample_seconds(x)
    out = {"value": x["kv_bytes"] / secs / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{n} of the {S} sequences (all {w.num_heads} heads, {int(x['lens'].sum())} tokens), "
                     f"new-token writes + fp64 attention, numpy single-threaded, {secs:.1f} s; tables and slots "
                     f"from the oracle's block manager"}
    if (os.cpu_count() or 1) > 1:
        out["all_cores"] = run_cpu_baseline_all_cores(args, seqs[:n])
    refs = None if args.no_configs else cpu_config_refs()
    return out, refs


def reference_sample(w):
    """The oracle arm's sequences per step: the whole batch, unless its K/V exceeds
    REF_MAX_KV_BYTES; then the longest sequences up to that many bytes."""
    if w.logical_kv_bytes() <= REF_MAX_KV_BYTES:
        return list(range(w.num_seqs)), f"the whole batch ({w.num_seqs} sequences, all {w.num_heads} heads)"
    per_token = w.num_heads * w.head_dim * 2 * 2
    seqs, total = [], 0
    for s in np.argsort(w.context_lens)[::-1]:
        b = int(w.context_lens[s]) * per_token
        if seqs and total + b > REF_MAX_KV_BYTES:
            break
        seqs.append(int(s))
        total += b
    return sorted(seqs), f"{len(seqs)} of the {w.num_seqs} sequences (the longest; the batch exceeds " \
                         f"{REF_MAX_KV_BYTES / 1e9:.1f} GB of K/V)"


def fit_reference_sample(w, seqs, step_s, runs, budget_s=REF_WALL_S):
    """The sequences of `seqs` (in order) the oracle arm keeps so that `runs` steps take about
    `budget_s` seconds, given that one step over all of `seqs` took `step_s`: a share of the K/V
    bytes in proportion, at least one sequence.  All of `seqs` when they fit."""
    if runs * step_s <= budget_s or len(seqs) <= 1:
        return list(seqs)
    keep = budget_s / (runs * step_s)
    lens = [int(w.context_lens[s]) for s in seqs]
    cap, out, acc = keep * sum(lens), [], 0
    for s, n in zip(seqs, lens):
        if out and acc + n > cap:
            break
        out.append(s)
        acc += n
    return out


def run_reference(args, rank):
    """The oracle, as it stands, on the host cores: each step the new-token writes and fp64
    attention over the batch, whose tables and slots the oracle's block manager builds."""
    if rank != 0:
        return None
    if args.workload in AUX_WORKLOADS:
        return {"impl": "reference", "unavailable": f"the oracle arm times the decode workloads, not {args.workload}"}
    seed = workload_seed(args.workload)
    x0 = build_step_inputs(seed, args.workload, args.capacity_seqs, args.capacity_block, manager="oracle")
    w = x0["w"]
    seqs, what = reference_sample(w)
    sample = prepare_cpu_sample(w, seqs, x0["slots"], x0["pairs"], seed)   # generated once, untimed
    # the first warm-up step also sizes the sample: the whole run stays within about REF_WALL_S
    runs = max(args.warmup, 1) + args.steps
    kept = fit_reference_sample(w, seqs, cpu_sample_seconds(sample), runs)
    if len(kept) < len(seqs):
        seqs = kept
        what = f"{len(seqs)} of the {w.num_seqs} sequences (all {w.num_heads} heads; sized so that {runs} " \
               f"steps take about {REF_WALL_S:.0f} s)"
        sample = prepare_cpu_sample(w, seqs, x0["slots"], x0["pairs"], seed)
        cpu_sample_seconds(sample)
    for _ in range(max(args.warmup, 1) - 1):
        cpu_sample_seconds(sample)
    secs = 0.0
    for _ in range(args.steps):
        secs += cpu_sample_seconds(sample)
    kv = sample["kv_bytes"] * args.steps
    value = kv / secs / 1e9
    desc = f"{what} per step: the step's copies, the new-token writes and fp64 attention (numpy, one thread); " \
           "tables and slots from the oracle's block manager"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-based generator)",
            "config": config_block(args, x0["desc"], w.num_seqs, flushed=needs_flush(w)),
            "same_config": len(seqs) == w.num_seqs,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---- the line --------------------------------------------------------------------------------------

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


def config_block(args, desc, num_seqs, flushed=False):
    """The workload the line is quoted on; the GPU arm and the oracle arm print the same block."""
    cfg_seed = workload_seed(args.workload)
    return {"workload": desc, "num_seqs": num_seqs,
            "num_heads": 2 if args.workload == "tiny" else 40, "head_dim": 64 if args.workload == "tiny" else 128,
            "block_size": args.capacity_block if args.workload == "capacity" else (4 if args.workload == "tiny" else 16),
            "seed": f"{cfg_seed} (+7919*rank)", "kv_storage": "f16",
            "l2": ("L2 flushed before every step (a write of twice the L2 size, outside the timed region); "
                   "each step timed by its own events") if flushed
            else "inputs larger than L2: the step reads more than twice the L2 size of distinct K/V"}


def reduce_run(r, world, device):
    """Whole-job figures of a run: times maxed over ranks, bytes summed over ranks."""
    loop = r.get("e2e_loop") or {}
    rep = r.get("e2e_replay") or {}
    sus = r.get("sustained") or {}
    names_t = ("step_ms", "attn_ms", "attn_ms_median", "e2e_s", "e2e_replay_ms", "e2e_staged_ms", "sus_s")
    vals_t = (r["step_ms"], r["attn_ms"], r["attn_ms_median"], loop.get("seconds", 0.0), rep.get("ms_per_step", 0.0),
              rep.get("staged_ms_per_step", 0.0), sus.get("device_s", 0.0))
    names_b = ("kv_total", "phys_total", "e2e_kv", "sus_kv")
    vals_b = (r["kv_bytes"], r["phys_bytes"], loop.get("kv_bytes", 0), sus.get("kv_bytes", 0))
    t, b = reduce_over_ranks(vals_t, [float(v) for v in vals_b], world, device)
    return dict(zip(names_t, t)) | dict(zip(names_b, b))


def headline_line(args, r, world, cpu, red):
    """The JSON line of a decode run: `r` is this rank's run_gpu result, `red` the whole-job
    figures (reduce_run)."""
    peak, peak_src = measured_hbm_peak()
    achieved = r["attn_bytes"] / (red["attn_ms"] * 1e-3) / 1e9
    traffic = None if args.grouped else NCU_TRAFFIC.get(
        (args.workload + ("+append" if r["fused"] else ""), attention_source_sha()))
    value = red["kv_total"] / (red["step_ms"] * 1e-3) / 1e9
    S = r["num_seqs"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": red["step_ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded counter-based generator)",
        "config": config_block(args, r["desc"], S, flushed=r["l2_flushed"]),
        "parallelism": f"replicas x{world} (each rank its own batch, no exchange)" if world > 1 else "single GPU",
        "plan": {"partition_tokens": r["part_tokens"], "kernels_per_step": r["kernels_per_step"],
                 "step": "fused" if r["fused"] else "unfused", "cow_pairs_per_step": r["n_pairs"],
                 "pool_blocks": r["num_blocks"]},
        "hbm_frac_of_measured": value / peak,
        "hbm_frac_of_nominal": value / NOMINAL_HBM_GBS,
        "physical_kv_GBps": red["phys_total"] / (red["step_ms"] * 1e-3) / 1e9,
        "tokens_per_s": S * world / (red["step_ms"] * 1e-3),
        "tokens_per_s_40_layer_attention_only": S * world / (40 * red["step_ms"] * 1e-3),
        "host_slot_assignment_us": r["host_slot_us"],
        "roofline": {"bound": "hbm",
                     "kernel": ("paged attention call with the new tokens' K/V append; bytes include the "
                                "appended rows read and written" if r["fused"]
                                else "paged attention call") if r["grouped"] is None
                     else "shared-prefix attention call (prefix partials on tensor cores + partition + merge); "
                          "bytes = distinct K/V slots + q + out",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": r["attn_bytes"],
                     "launch_ms": red["attn_ms"], "launch_ms_median_isolated": red["attn_ms_median"],
                     "timed_launches": r["timed_launches"], "launch_timing": r["attn_loop"],
                     "peak_source": peak_src + ", of measured"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "clocks_timed_region": r["clocks_timed_region"],
    }
    if r.get("sustained"):
        s = r["sustained"]
        sv = red["sus_kv"] / red["sus_s"] / 1e9 if red["sus_s"] > 0 else None
        mhz = (s.get("clocks") or {}).get("sm_mhz")
        line["sustained"] = {"value": sv, "unit": UNIT, "steps": s["steps"], "seconds": s["seconds"],
                             "ms_per_step": s["ms_per_step"], "clocks": s["clocks"],
                             "ms_x_median_sm_mhz": None if mhz is None else s["ms_per_step"] * mhz}
    if r["copy"] is not None:
        line["copy_blocks_setup"] = r["copy"]
    if r.get("bm") is not None:
        line["block_manager"] = r["bm"]
    if r["grouped"] is not None:
        line["grouped"] = r["grouped"]
    loop, rep = r.get("e2e_loop"), r.get("e2e_replay")
    if loop and "seconds" in loop:
        e2e = {"value": red["e2e_kv"] / red["e2e_s"] / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": loop["h2d_bytes_per_step"], "d2h_bytes_per_step": loop["d2h_bytes_per_step"],
               "ms_per_step": loop["ms_per_step"], "steps": loop["steps"],
               "host_a1_us_per_step": loop["host_a1_us_per_step"], "copies": loop["copies"],
               "launch": ("every step pkv_bm_append_slots + pkv_bm_block_tables write the step's slots, tables and "
                          "lengths into page-locked host memory (the next step's into a second buffer set while this "
                          "step's kernels run), the kernels read them and q and the new K/V rows across NVLink-C2C "
                          "and write the output there, the host waits for it; contexts grow by one token a step; "
                          "device calls: " + loop.get("launch_form", "eager C-ABI calls")) if not loop["staged"]
               else ("every step pkv_bm_append_slots + pkv_bm_block_tables (the next step's beside this step's "
                     "kernels), one copy of the step's inputs to the device and of the output back, the host "
                     "waits; contexts grow by one token a step")}
        if rep:
            e2e["graph_replay"] = {"value": red["kv_total"] / (red["e2e_replay_ms"] * 1e-3) / 1e9,
                                   "ms_per_step": rep["ms_per_step"], "launch": rep["launch"],
                                   "staged_value": red["kv_total"] / (red["e2e_staged_ms"] * 1e-3) / 1e9,
                                   "staged_ms_per_step": rep["staged_ms_per_step"],
                                   "h2d_bytes_per_step": rep["h2d_bytes_per_step"]}
        line["e2e"] = e2e
    elif loop:
        line["e2e"] = {"value": None, "unit": UNIT, "skipped": loop.get("skipped")}
    if r.get("configs") is not None:
        line["configs"] = r["configs"]
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

    cpu, refs = None, None
    if rank == 0 and not args.no_cpu_baseline and args.workload not in AUX_WORKLOADS:
        cpu, refs = run_cpu_baseline(args)                # before any GPU work: the oracle runs alone

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from paged_kv_cache_73_gb300 import binding as pkv
    pkv.load()
    if args.workload in AUX_WORKLOADS:
        line = {"swap": run_swap, "layers40": run_layers40, "prefill": run_prefill}[args.workload](args, dev)
        if rank == 0:
            print(json.dumps(line), flush=True)
    else:
        r = run_gpu(args, rank, world, dev, refs)
        red = reduce_run(r, world, dev)                   # whole job: all ranks' bytes over the slowest rank
        if rank == 0:
            print(json.dumps(headline_line(args, r, world, cpu, red)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
