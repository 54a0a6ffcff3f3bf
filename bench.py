"""Benchmark: one decode step of one layer over a block-paged KV cache.

A step is the whole hot path over one batch: address translation of the
step's new tokens and their K/V append in one launch (paged_kv_append_tokens,
which computes what paged_kv_slot_mapping + paged_kv_append do) and the fused
paged-attention decode of every sequence (paged_attention_decode, split-K
partitions + merge where configured).

Default workload: the long-context layer, the largest that fits one GPU (8
sequences, lengths uniform in [32768, 131072], 64 q / 8 kv heads, head_dim
128, bf16, block size 16, 512-token partitions + LSE merge), synthetic seeded
inputs. The GQA batch-256 and MHA layers, the continuous-batching trace and
the next rows (copy-on-write, swap, chunked prefill) are measured after it.

Prints one JSON line (rank 0). `value` is whole-job paged-decode GB/s: the
step's algorithmic bytes (unique KV bytes + q + out + block-table + length
bytes) over the device-timed step; `roofline` is the decode call alone, timed
back to back. The line ends with `targets`, the compact per-workload decode
fractions of the measured HBM peak. `--impl reference` times the fp64 CPU
oracle instead on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import materialize, new_pools, preset, subset  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak); seq-decodes/s per layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129e6
KERNEL_SOURCES = ["decode_kernel.cuh", "decode_params.h", "ptx.cuh", "merge.cu", "api.cu",
                  "decode_instances.cuh", "decode_launch.h", "launch_cache.h"]

# partition size (tokens) used for each workload's decode; 0 = no split, -1 the
# balanced split (equal tile shares per CTA). Measured on GB300, back to back,
# with the decode's L2 priorities (shared blocks evict_last, the rest
# evict_first): the MHA layer is fastest with the balanced split (0.992 of the
# copy peak; 0.925 with 192-token partitions, the best fixed size, before the
# priorities); the GQA layer with the balanced split too (0.944 with its
# three-stage ring; 320-token partitions, the best fixed size, 0.869-0.882,
# reported beside it under the shared-prefix entry's figures; without the
# priorities the balanced split's contiguous shares read each group's shared
# prefix at times too far apart for L2, 0.787); the long-context workload
# states its 512-token partitions (0.989; the balanced split is reported
# beside it).
PARTITION = {"tiny": 0, "mha7b": -1, "gqa8b_prefix": -1, "longctx_splitk": 512}

DESCRIPTION = {
    "tiny": "tiny: 4 seqs, lens {2,18,34,65}, B16, 4q/2kv heads, D64, fp32",
    "mha7b": "mha7b: Llama-2-7B-shaped MHA layer, 64 seqs, lens U[128,2048], 32q=32kv heads, "
             "D128, fp16, B16, shuffled pool 1.25x need",
    "gqa8b_prefix": "gqa8b_prefix: Llama-3-8B-shaped GQA layer, 256 seqs, lognormal lens "
                    "(median 1024, sigma 0.75, clip [513,8192]), 32q/8kv heads, D128, bf16, B16, "
                    "groups of 16 share a 512-token prefix",
    "longctx_splitk": "longctx_splitk: 8 seqs, lens U[32768,131072], 64q/8kv heads, D128, bf16, "
                      "B16, 512-token partitions + LSE merge",
}


# ---------------------------------------------------------------------------
# Byte accounting (algorithmic: what the method must move at minimum)
# ---------------------------------------------------------------------------

def decode_bytes(wl):
    """(algorithmic bytes per decode, logical-KV bytes per decode, KV-unique bytes)."""
    B, elt = wl.block_size, wl.element_bytes
    row = wl.n_kv_heads * wl.head_dim * elt          # one token's K (or V) for all kv heads
    used = {}
    nblk_total = 0
    for s in range(wl.num_seqs):
        L = int(wl.context_lens[s])
        nb = -(-L // B)
        nblk_total += nb
        for j in range(nb):
            b = int(wl.block_tables[s, j])
            n = min(B, L - j * B)
            if used.get(b, 0) < n:
                used[b] = n
    kv_unique = 2 * row * sum(used.values())
    kv_logical = 2 * row * int(wl.context_lens.sum())
    other = 2 * wl.num_seqs * wl.n_q_heads * wl.head_dim * elt + 4 * nblk_total + 4 * wl.num_seqs
    return kv_unique + other, kv_logical + other, kv_unique


def append_bytes(wl, tokens):
    return 2 * 2 * tokens * wl.row_bytes + 8 * tokens


def measured_peak():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense 16-bit tensor TFLOP/s of this GPU: the burst figure (a kernel timed alone)."""
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def decode_part_of_api(text):
    """The parts of api.cu that decide a decode launch: the options' defaults,
    the pool tensor map, the workspace layout and the decode entry points (other
    entry points excluded)."""
    try:
        a = text.index("int encode_pool_map(")
        b = text.index("size_t round256(")
        c = text.index("size_t paged_attention_workspace_bytes(")
    except ValueError:
        return text
    options = "".join(line for line in text.splitlines(True) if line.startswith("int g_opt_"))
    return options + text[a:b] + text[c:]


def code_only(text):
    """C/C++ source without its comments and blank lines (string and character
    literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_digest():
    """Digest of the code (comments aside) that determines the decode kernels
    and their launch."""
    h = hashlib.sha256()
    csrc = os.path.join(REPO, "paged_kv_cache_233_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        if name == "api.cu":
            text = decode_part_of_api(text)
        h.update(code_only(text).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload, partition):
    """DRAM bytes per decode launch from a committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(REPO, "profiles", f"decode_{workload}_traffic.txt")
    try:
        kv = dict(line.strip().split("=", 1) for line in open(path) if "=" in line)
    except OSError:
        return None
    if kv.get("source_digest") != kernel_source_digest() or int(kv.get("partition", -1)) != partition:
        return None
    try:
        return float(kv["dram_bytes_per_decode"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# The step
# ---------------------------------------------------------------------------

class Step:
    """Device-resident inputs and the two calls of one decode step: the new
    tokens' slot mapping and append in one launch, then the decode."""

    def __init__(self, wl, device, partition):
        import paged_kv_cache_233_gb300 as pk
        self.pk = pk
        self.wl = wl
        self.partition = partition
        self.t = materialize(wl, device)
        self.kc, self.vc = new_pools(wl, device, fill=0.0)
        self.bt = torch.from_numpy(wl.block_tables).to(device)
        self.lens = torch.from_numpy(wl.context_lens).to(device)
        self.step_seq = torch.from_numpy(wl.step_seq).to(device)
        self.step_pos = torch.from_numpy(wl.step_pos).to(device)
        self.slots = torch.empty(len(wl.step_seq), dtype=torch.int64, device=device)
        self.out = torch.empty_like(self.t["q"])
        self.ws = pk.new_workspace(self.t["q"], self.bt, wl.block_size, partition)
        # bulk fill of the history (timed separately: append GB/s over the whole context)
        fill_seq = torch.from_numpy(wl.fill_seq).to(device)
        fill_pos = torch.from_numpy(wl.fill_pos).to(device)
        fill_slots = torch.empty(len(wl.fill_seq), dtype=torch.int64, device=device)
        pk.paged_kv_slot_mapping(self.bt, fill_seq, fill_pos, fill_slots, wl.num_blocks,
                                 wl.block_size)
        # one untimed fill (the first launch of the kernel in the process carries
        # one-time costs), then the median of three timed fills of the same rows
        # into the same slots (each writes the same bytes)
        pk.paged_kv_append(self.t["k_fill"], self.t["v_fill"], fill_slots, self.kc, self.vc)
        torch.cuda.synchronize()
        fills = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pk.paged_kv_append(self.t["k_fill"], self.t["v_fill"], fill_slots, self.kc, self.vc)
            e1.record()
            torch.cuda.synchronize()
            fills.append(e0.elapsed_time(e1))
        self.fill_ms = statistics.median(fills)
        self.fill_tokens = len(wl.fill_seq)
        del fill_seq, fill_pos, fill_slots
        self.launches_per_step = 2 + (1 if partition != 0 else 0)   # the merge of a split

    def run(self):
        self.pk.paged_kv_append_tokens(self.t["k_step"], self.t["v_step"], self.bt, self.step_seq,
                                       self.step_pos, self.kc, self.vc)
        self.decode()

    def decode(self):
        self.pk.paged_attention_decode(self.t["q"], self.kc, self.vc, self.bt, self.lens,
                                       self.wl.scale, self.out, self.partition, self.ws)

    def use_shared_prefix_entry(self):
        """Decode through paged_attention_decode_shared_prefix with the
        workload's prefix groups (consecutive members sharing their first
        prefix_blocks blocks)."""
        wl, dev = self.wl, self.out.device
        seq_group = np.full(wl.num_seqs, -1, np.int32)
        for gi, grp in enumerate(wl.groups):
            seq_group[grp] = gi
        self.seq_group = torch.from_numpy(seq_group).to(dev)
        self.group_prefix = torch.full((max(1, len(wl.groups)),), wl.prefix_blocks * wl.block_size,
                                       dtype=torch.int32, device=dev)

        def decode():
            self.pk.paged_attention_decode_shared_prefix(
                self.t["q"], self.kc, self.vc, self.bt, self.lens, self.seq_group,
                self.group_prefix, self.wl.scale, self.out, self.partition, self.ws)
        self.decode = decode


def time_steps(step, steps, dist_ctx):
    """Device time of exactly `steps` steps between one pair of events (no
    event between the launches, which would end their programmatic dependent
    overlap), max over ranks."""
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_ctx.barrier()
    torch.cuda.synchronize()
    start.record()
    for _ in range(steps):
        step.run()
    stop.record()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    return dist_ctx.max(start.elapsed_time(stop))


def time_decode_calls(call, reps, repeats=5):
    """`reps` decode calls back to back between one pair of events, `repeats`
    times; returns the mean ms per call of each repeat. Back to back, a call's
    set-up overlaps the previous call's tail, as along a serving step."""
    out = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / reps)
    return out


def time_each_call(call, reps):
    """Median ms of `reps` decode calls, each bracketed by its own events."""
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in pairs:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in pairs)


_FLUSH = {}


def time_each_call_l2_flushed(call, reps=30):
    """Median ms of `reps` decode calls, each bracketed by its own events after
    a write of twice the L2's bytes (nothing a call read is left in L2 for the
    next one: the cold-cache time of one call)."""
    dev = torch.cuda.current_device()
    if dev not in _FLUSH:
        _FLUSH[dev] = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device="cuda")
    buf = _FLUSH[dev]
    times = []
    for _ in range(reps):
        buf.fill_(1.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def spread(xs):
    """min / median / max of repeated measurements and the max-min range in % of the median."""
    med = statistics.median(xs)
    return {"n": len(xs), "min": min(xs), "median": med, "max": max(xs),
            "range_pct": 100.0 * (max(xs) - min(xs)) / med if med else None}


E2E_INPUTS = ("q", "k", "v", "bt", "lens", "seq", "pos")


def e2e_sources(step, q=None):
    """The step's seven input arrays (q replaced by `q` when given)."""
    t = step.t
    return dict(zip(E2E_INPUTS, (t["q"] if q is None else q, t["k_step"], t["v_step"], step.bt,
                                 step.lens, step.step_seq, step.step_pos)))


def pack_host_inputs(src):
    """One pinned host buffer holding every input array of a step, each on a
    256-byte boundary; returns (buffer, offsets)."""
    offs, size = {}, 0
    for n in E2E_INPUTS:
        offs[n] = size
        size += (src[n].numel() * src[n].element_size() + 255) // 256 * 256
    host = torch.empty(size, dtype=torch.uint8).pin_memory()
    for n in E2E_INPUTS:
        x = src[n].contiguous().cpu()
        nb = x.numel() * x.element_size()
        host[offs[n]:offs[n] + nb].copy_(x.view(-1).view(torch.uint8))
    return host, offs


def time_e2e(step, steps, host_inputs=None, outputs=None):
    """Same step through the public API with host inputs: every step copies its
    inputs from pinned host memory to the device and reads its output back.

    The step's seven input arrays are packed in one pinned host buffer and
    copied with one transfer into one of two device staging buffers; the copy
    of step i+1 and the read-back of step i run on a copy stream while step i
    computes (double-buffered inputs and outputs), as a serving loop would
    overlap them. Step i takes host_inputs[i % len(host_inputs)] (by default
    one buffer of the step's own inputs) and, when `outputs` (a list of pinned
    host tensors, one per step) is given, reads back into outputs[i] instead
    of the two alternating host buffers."""
    wl = step.wl
    src = e2e_sources(step)
    if host_inputs is None:
        host_inputs = [pack_host_inputs(src)[0]]
    offs, size = {}, 0
    for n in E2E_INPUTS:
        offs[n] = size
        size += (src[n].numel() * src[n].element_size() + 255) // 256 * 256
    dev = [torch.empty(size, dtype=torch.uint8, device=step.out.device) for _ in range(2)]

    def views(buf):
        v = {}
        for n in E2E_INPUTS:
            x = src[n]
            nb = x.numel() * x.element_size()
            v[n] = buf[offs[n]:offs[n] + nb].view(x.dtype).view(x.shape)
        return v

    vs = [views(d) for d in dev]
    outs = [step.out, torch.empty_like(step.out)]
    out_host = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(src[n].numel() * src[n].element_size() for n in E2E_INPUTS)
    d2h = out_host[0].numel() * out_host[0].element_size()
    pk = step.pk
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def run(v, out):
        pk.paged_kv_append_tokens(v["k"], v["v"], v["bt"], v["seq"], v["pos"], step.kc, step.vc)
        pk.paged_attention_decode(v["q"], step.kc, step.vc, v["bt"], v["lens"], wl.scale, out,
                                  step.partition, step.ws)

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    copy.wait_stream(compute)
    with torch.cuda.stream(copy):
        dev[0].copy_(host_inputs[0], non_blocking=True)
        ready[0].record(copy)
    for i in range(steps):
        b = i % 2
        compute.wait_event(ready[b])
        run(vs[b], outs[b])
        done[b].record(compute)
        with torch.cuda.stream(copy):
            if i + 1 < steps:
                if i >= 1:
                    copy.wait_event(done[1 - b])       # step i-1 no longer reads that buffer
                dev[1 - b].copy_(host_inputs[(i + 1) % len(host_inputs)], non_blocking=True)
                ready[1 - b].record(copy)
            copy.wait_event(done[b])
            dst = outputs[i] if outputs is not None else out_host[b]
            dst.copy_(outs[b], non_blocking=True)
    compute.wait_stream(copy)
    e1.record(compute)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ---------------------------------------------------------------------------

def host_storage(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_pools(orc, wl, tensors):
    shape = (wl.num_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim)
    np_dtype = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[wl.dtype]
    kc = np.zeros(shape, dtype=np_dtype)
    vc = np.zeros(shape, dtype=np_dtype)
    for seq, pos, k, v in ((wl.fill_seq, wl.fill_pos, tensors["k_fill"], tensors["v_fill"]),
                           (wl.step_seq, wl.step_pos, tensors["k_step"], tensors["v_step"])):
        sm = orc.slot_mapping(wl.block_tables, seq, pos, wl.block_size)
        orc.append(host_storage(k), host_storage(v), sm, kc, vc)
    return kc, vc


# sequences of each workload the CPU oracle is timed on (a bounded sample: its
# pools and inputs are built on the host for these sequences only)
ORACLE_SAMPLE_SEQS = {"tiny": None, "mha7b": None, "gqa8b_prefix": list(range(32)),
                      "longctx_splitk": [0, 1]}


def oracle_sample(orc, name):
    """The workload (or its sampled sequences) with host q and oracle-filled pools."""
    wl = preset(name)
    seqs = ORACLE_SAMPLE_SEQS.get(name)
    if seqs is not None:
        wl = subset(wl, seqs)
    tensors = materialize(wl, "cpu")
    kc, vc = oracle_pools(orc, wl, tensors)
    return wl, host_storage(tensors["q"]), kc, vc


def oracle_rate(orc, wl, q, kc, vc, budget_s, start_unit=0, threads=None):
    """Time the oracle's decode over consecutive (seq, kv head) units, cycling
    through the workload, until the budget is spent (all host cores unless
    `threads` is given). Returns (bytes, seconds, units, threads)."""
    units = [(s, h) for s in range(wl.num_seqs) for h in range(wl.n_kv_heads)]
    threads = threads or orc.max_threads()
    row = wl.head_dim * wl.element_bytes
    done_bytes, elapsed, n = 0, 0.0, 0
    i = start_unit % len(units)
    chunk = max(1, threads)
    while elapsed < budget_s:
        batch = [units[(i + k) % len(units)] for k in range(chunk)]
        t0 = time.perf_counter()
        orc.decode(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, units=batch,
                   threads=threads)
        elapsed += time.perf_counter() - t0
        for s, _ in batch:
            L = int(wl.context_lens[s])
            done_bytes += 2 * L * row + 2 * wl.group * wl.head_dim * wl.element_bytes
        n += len(batch)
        i += len(batch)
    return done_bytes, elapsed, n, threads


# ---------------------------------------------------------------------------
# Distributed plumbing (one process per GPU; replicas of the workload)
# ---------------------------------------------------------------------------

class DistCtx:
    def __init__(self, connect=True):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1 and connect:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x):
        if self.pg is None:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x):
        if self.pg is None:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def workload_config(name, wl, partition, world):
    """The `config` object of the JSON line, the same for both arms."""
    pool = 2 * wl.num_blocks * wl.block_size * wl.row_bytes
    return {"workload": DESCRIPTION[name] if wl.name == name else wl.name,
            "partition_tokens": partition,
            "l2": (f"inputs {'larger' if pool > L2_BYTES else 'smaller'} than L2: "
                   f"KV pool {pool / 1e9:.2f} GB"),
            "parallelism": f"replicas x{world} (one workload per GPU)"}


def workload_for(name, rank):
    wl = preset(name)
    if rank:
        wl = preset(name, seed=wl.seed + 1000 * rank)
    return wl


# ---------------------------------------------------------------------------
# Arms
# ---------------------------------------------------------------------------

def run_reference(args, ctx):
    """The fp64 CPU oracle, as it stands, on bounded samples of the workload."""
    if ctx.rank != 0:
        return None
    import oracle
    orc = oracle.get()
    wl, q, kc, vc = oracle_sample(orc, args.config)
    per_step = max(0.05, min(20.0, args.reference_budget / max(1, args.steps + args.warmup)))
    for w in range(args.warmup):
        oracle_rate(orc, wl, q, kc, vc, per_step, start_unit=w)
    total_bytes, total_s, total_units, threads = 0, 0.0, 0, 1
    for k in range(args.steps):
        b, s, n, threads = oracle_rate(orc, wl, q, kc, vc, per_step, start_unit=k * 7)
        total_bytes += b
        total_s += s
        total_units += n
    value = total_bytes / total_s / 1e9
    sample = (f"{total_units} (sequence, kv head) units of {wl.name} over {args.steps} steps, "
              f"~{per_step:.2f} s of oracle work per step, of {wl.num_seqs * wl.n_kv_heads} units")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": ctx.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(args.config, preset(args.config), PARTITION[args.config], ctx.world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def decode_figures(wl, call, reps, repeats=5):
    """Decode-call figures of one workload: the median of `reps` calls each
    between its own events, the median of 30 such calls each after an L2
    flush, and `repeats` runs of `reps` calls back to back."""
    algo, logical, kv_unique = decode_bytes(wl)
    peak, _ = measured_peak()
    per_call = time_each_call(call, reps)
    flushed = time_each_call_l2_flushed(call)
    b2b = time_decode_calls(call, reps, repeats)
    med = statistics.median(b2b)
    return {"algorithmic_bytes": algo, "kv_unique_bytes": kv_unique,
            "decode_ms_back_to_back": med, "back_to_back_ms_spread": spread(b2b),
            "achieved_gbs": algo / med / 1e6, "frac": algo / med / 1e6 / peak,
            "logical_gbs": logical / med / 1e6,
            "decode_ms_per_call": per_call, "frac_per_call": algo / per_call / 1e6 / peak,
            "decode_ms_l2_flushed": flushed, "frac_l2_flushed": algo / flushed / 1e6 / peak,
            "reps": reps}


def measure_gate(name, args, device, partition=None):
    """Decode-only roofline fraction of one workload (for the stated targets)."""
    import paged_kv_cache_233_gb300 as pk
    wl = preset(name)
    P = PARTITION[name] if partition is None else partition
    step = Step(wl, device, P)
    for _ in range(args.warmup):
        step.run()
    res = decode_figures(wl, step.decode, args.gate_reps)
    res.update(partition_tokens=P, decode_path=pk.last_decode_path())
    del step
    torch.cuda.empty_cache()
    return res


TRACE_SLOTS = (8, 16, 32, 64, 128, 256)


def trace_bytes(tw, plans):
    """(decode algorithmic bytes, append bytes, sequence-decodes) of the trace's steps."""
    from types import SimpleNamespace
    dec_bytes = app_bytes = decodes = 0
    row = tw.n_kv_heads * tw.head_dim * tw.element_bytes
    for plan in plans:
        view = SimpleNamespace(block_size=tw.block_size, element_bytes=tw.element_bytes,
                               n_kv_heads=tw.n_kv_heads, head_dim=tw.head_dim,
                               n_q_heads=tw.n_q_heads, num_seqs=len(plan.rids),
                               context_lens=plan.context_lens, block_tables=plan.block_tables)
        dec_bytes += decode_bytes(view)[0]
        app_bytes += 4 * len(plan.token_row) * row + 8 * len(plan.token_row)
        decodes += len(plan.rids)
    return dec_bytes, app_bytes, decodes


class TraceRun:
    """The continuous-batching workload's steps, ready on the device: per step
    the appended tokens' K/V rows and (row, position) pairs, the block tables,
    lengths and queries, and an output buffer; one workspace for every step, as
    a serving loop keeps it. run_pass() issues every step's
    paged_kv_append_tokens and paged_attention_decode on the current stream."""

    def __init__(self, tw, device, partition, pools=None):
        import paged_kv_cache_233_gb300 as pk
        from workloads import step_inputs, trace_tensors
        self.pk, self.tw, self.partition = pk, tw, partition
        tensors = trace_tensors(tw, device)
        shape = (tw.num_blocks, tw.block_size, tw.n_kv_heads, tw.head_dim)
        if pools is None:
            pools = (torch.zeros(shape, dtype=tw.torch_dtype, device=device),
                     torch.zeros(shape, dtype=tw.torch_dtype, device=device))
        self.kc, self.vc = pools
        self.steps = []
        ws_bytes = 0
        for plan in tw.plans:
            x = step_inputs(tw, plan, tensors, device)
            x["out"] = torch.empty_like(x["q"])
            q, bt = x["q"], x["block_tables"]
            ws_bytes = max(ws_bytes, pk.paged_attention_workspace_bytes(
                q.shape[0], q.shape[1], q.shape[2], bt.shape[1], tw.block_size, partition))
            self.steps.append((plan, x))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device) if ws_bytes else None

    def run_pass(self, ev=None):
        pk, tw = self.pk, self.tw
        for i, (plan, x) in enumerate(self.steps):
            if ev is not None:
                ev[i][0].record()
            pk.paged_kv_append_tokens(x["k"], x["v"], x["block_tables"], x["token_row"],
                                      x["token_pos"], self.kc, self.vc)
            pk.paged_attention_decode(x["q"], self.kc, self.vc, x["block_tables"],
                                      x["context_lens"], tw.scale, x["out"], self.partition,
                                      self.ws)
            if ev is not None:
                ev[i][1].record()

    def capture(self):
        """The whole pass captured in one CUDA graph (run one pass eagerly first,
        so that every kernel's launch attributes are already set)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self.run_pass()
        return g


def measure_trace(block_size, device, slots=64, partition=None, passes=5, pool_tokens=65536):
    """The continuous-batching workload (64 requests, up to `slots` running,
    65,536-slot pool, LIFO recompute preemption) through the hot path, step by
    step: each step one paged_kv_append_tokens and one paged_attention_decode
    (TraceRun).

    Two ways of issuing the same launches, after one untimed pass:
      graph  the whole pass captured once in a CUDA graph and replayed, so the
             device runs the steps back to back, as a serving loop that
             captures its decode step does; `passes` replays, each between
             its own events (the headline figures: the device's time);
      eager  the steps issued one by one from Python through the binding,
             each step between its own events (`passes` passes; the pass of
             median total time), bounded by the host's issue rate when the
             device is faster than the host.
    The trace's contexts are short (<= 640 tokens) and its batches small
    (<= 32 running), so a step's decode runs the balanced split."""
    import paged_kv_cache_233_gb300 as pk
    if partition is None:
        partition = pk.PARTITION_BALANCED
    from workloads import cb_trace
    tw = cb_trace(block_size=block_size, slots=slots, pool_tokens=pool_tokens)
    tr = TraceRun(tw, device, partition)
    tr.run_pass()
    torch.cuda.synchronize()
    plans = [p for p, _ in tr.steps]
    dec_bytes, app_bytes, decodes = trace_bytes(tw, plans)
    res = {"slots": slots, "pool_tokens": pool_tokens, "steps": len(plans),
           "preemptions": tw.preemptions,
           "max_running": max(len(p.rids) for p in plans), "partition_tokens": partition,
           "decode_bytes": dec_bytes}
    graph_ms = None
    try:
        g = tr.capture()
        g.replay()
        torch.cuda.synchronize()
        runs = []
        for _ in range(passes):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            runs.append(e0.elapsed_time(e1))
        graph_ms = statistics.median(runs)
        res.update({"total_ms": graph_ms, "decode_gbs": dec_bytes / graph_ms / 1e6,
                    "seq_decodes_per_s": decodes / (graph_ms * 1e-3),
                    "append_gbs_in_step": app_bytes / graph_ms / 1e6,
                    "mean_step_us": 1e3 * graph_ms / len(plans), "issued": "one CUDA graph",
                    "pass_ms_spread": spread(runs)})
        del g
    except RuntimeError as exc:   # report, then time eagerly only
        res["graph_error"] = str(exc)[:200]
    runs = []
    for _ in range(passes):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in plans]
        tr.run_pass(ev)
        torch.cuda.synchronize()
        runs.append([a.elapsed_time(b) for a, b in ev])
    ms = sorted(runs, key=sum)[len(runs) // 2]
    eager_ms = sum(ms)
    res["eager"] = {"total_ms": eager_ms, "decode_gbs": dec_bytes / eager_ms / 1e6,
                    "median_step_us": 1e3 * statistics.median(ms),
                    "pass_ms_range": [min(map(sum, runs)), max(map(sum, runs))]}
    if graph_ms is None:
        res.update({"total_ms": eager_ms, "decode_gbs": dec_bytes / eager_ms / 1e6,
                    "seq_decodes_per_s": decodes / (eager_ms * 1e-3),
                    "append_gbs_in_step": app_bytes / eager_ms / 1e6, "issued": "eager"})
    assert pk.device_errors() == 0
    del tr
    torch.cuda.empty_cache()
    return res


def measure_shared_prefix(device, reps=200, partitions=(256, 320, 512)):
    """The GQA prefix workload through paged_attention_decode_shared_prefix
    (each whole prefix partition read once per chunk of members instead of
    once per member), against the same roofline numerator as the plain decode,
    with the plain decode at the same partition size beside it."""
    import paged_kv_cache_233_gb300 as pk
    wl = preset("gqa8b_prefix")
    seq_group = np.full(wl.num_seqs, -1, np.int32)
    for gi, grp in enumerate(wl.groups):
        seq_group[grp] = gi
    res = {}
    for P in partitions:
        step = Step(wl, device, P)
        sg = torch.from_numpy(seq_group).to(device)
        gp = torch.full((len(wl.groups),), wl.prefix_blocks * wl.block_size, dtype=torch.int32,
                        device=device)

        def call():
            pk.paged_attention_decode_shared_prefix(step.t["q"], step.kc, step.vc, step.bt,
                                                    step.lens, sg, gp, wl.scale, step.out, P,
                                                    step.ws)
        for _ in range(5):
            call()
            step.decode()
        shared = decode_figures(wl, call, reps, repeats=3)
        plain = decode_figures(wl, step.decode, reps, repeats=3)
        res[f"P{P}"] = {"shared_prefix_entry": shared, "plain_decode": plain}
        del step
        torch.cuda.empty_cache()
    return res


def measure_cow(device, samples=4, reps=50):
    """Copy-on-write block copies of parallel sampling over the bench workload:
    every sequence of the MHA layer forks `samples` samples, and each sample's
    first token copies the sequence's shared last block to a fresh block."""
    import paged_kv_cache_233_gb300 as pk
    wl = preset("mha7b")
    shape = (wl.num_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim)
    kc = torch.zeros(shape, dtype=wl.torch_dtype, device=device)
    vc = torch.zeros_like(kc)
    used = set(wl.blocks_in_use().tolist())
    free = [b for b in range(wl.num_blocks) if b not in used]
    pairs = []
    for s in range(wl.num_seqs):
        last = int(wl.block_tables[s, (int(wl.context_lens[s]) - 1) // wl.block_size])
        for _ in range(samples):
            if free:
                pairs.append([last, free.pop()])
    pr = torch.tensor(pairs, dtype=torch.int32, device=device)
    for _ in range(3):
        pk.paged_kv_copy_blocks(kc, vc, pr)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        pk.paged_kv_copy_blocks(kc, vc, pr)
        b.record()
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    block_bytes = wl.block_size * wl.row_bytes
    moved = 2 * 2 * len(pairs) * block_bytes          # K and V, read + write
    del kc, vc
    torch.cuda.empty_cache()
    return {"pairs": len(pairs), "bytes_moved": moved, "median_us": ms * 1e3,
            "gbs": moved / ms / 1e6}


def measure_swap(device, reps=20):
    """Swap preemption over the bench workload: the blocks of a quarter of the
    MHA layer's sequences go out to a pinned host pool and back in, one call per
    direction. Compared with the copy engine moving the same bytes as one
    contiguous copy between the same kinds of memory (the link's practical rate)."""
    import paged_kv_cache_233_gb300 as pk
    wl = preset("mha7b")
    shape = (wl.num_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim)
    kc = torch.randn(shape, device=device).to(wl.torch_dtype)
    vc = torch.randn(shape, device=device).to(wl.torch_dtype)
    victims = range(0, wl.num_seqs, 4)
    src = np.concatenate([wl.block_tables[s][wl.block_tables[s] >= 0] for s in victims])
    n = len(src)
    hk = torch.empty((n,) + shape[1:], dtype=wl.torch_dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    host_ids = np.arange(n, dtype=np.int32)
    out_pairs = torch.from_numpy(np.stack([src, host_ids], 1).astype(np.int32)).to(device)
    in_pairs = torch.from_numpy(np.stack([host_ids, src], 1).astype(np.int32)).to(device)
    block_bytes = wl.block_size * wl.row_bytes
    moved = 2 * n * block_bytes                        # K and V blocks across the link

    def timed(fn):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    out_ms = timed(lambda: pk.paged_kv_swap_blocks(kc, vc, hk, hv, out_pairs))
    in_ms = timed(lambda: pk.paged_kv_swap_blocks(hk, hv, kc, vc, in_pairs))
    dev_buf = torch.empty(moved, dtype=torch.uint8, device=device)
    host_buf = torch.empty(moved, dtype=torch.uint8).pin_memory()
    ce_out_ms = timed(lambda: host_buf.copy_(dev_buf, non_blocking=True))
    ce_in_ms = timed(lambda: dev_buf.copy_(host_buf, non_blocking=True))
    assert pk.device_errors() == 0
    del kc, vc, dev_buf
    torch.cuda.empty_cache()
    res = {"blocks": int(n), "bytes_per_direction": int(moved),
           "out_us": out_ms * 1e3, "in_us": in_ms * 1e3,
           "out_gbs": moved / out_ms / 1e6, "in_gbs": moved / in_ms / 1e6,
           "copy_engine_out_gbs": moved / ce_out_ms / 1e6,
           "copy_engine_in_gbs": moved / ce_in_ms / 1e6}
    res["out_frac_of_copy_engine"] = res["out_gbs"] / res["copy_engine_out_gbs"]
    res["in_frac_of_copy_engine"] = res["in_gbs"] / res["copy_engine_in_gbs"]
    return res


def prefill_flops(context_lens, query_start, n_q_heads, head_dim):
    """4 * D per (query row, query head, key attended): Q K^T and P V, causal."""
    total = 0
    for s in range(len(context_lens)):
        n = int(query_start[s + 1] - query_start[s])
        L = int(context_lens[s])
        # rows attend over L - n + 1 .. L keys
        total += n * (L - n + 1) + n * (n - 1) // 2
    return 4 * head_dim * n_q_heads * total


def measure_prefill(device, reps=50, chunked=True):
    """Chunked-prefill attention: (1) a step of 16 Llama-2-7B-layer sequences
    each appending a 512-token chunk after U[0, 3584] cached tokens; (2) the
    serving page's scenario, one 2048-token prompt prefilled in one pass or in
    chunks of 512, 256 or 128 tokens (attention time of the whole prompt)."""
    import paged_kv_cache_233_gb300 as pk
    from workloads import chunked_prefill, prefill_mha7b, prefill_queries
    peak, peak_kind = measured_tensor_peak()

    def fill_pools(wl, dev):
        """Pools holding every token of the workload, written by slot mapping + append."""
        t = materialize(wl, dev)
        kc, vc = new_pools(wl, dev, fill=0.0)
        bt = torch.from_numpy(wl.block_tables).to(dev)
        for seq, pos, k, v in ((wl.fill_seq, wl.fill_pos, t["k_fill"], t["v_fill"]),
                               (wl.step_seq, wl.step_pos, t["k_step"], t["v_step"])):
            slots = torch.empty(len(seq), dtype=torch.int64, device=dev)
            pk.paged_kv_slot_mapping(bt, torch.from_numpy(seq).to(dev),
                                     torch.from_numpy(pos).to(dev), slots, wl.num_blocks,
                                     wl.block_size)
            pk.paged_kv_append(k, v, slots, kc, vc)
        return kc, vc, bt

    def timed(fn, n=reps):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    wl, qs = prefill_mha7b()
    kc, vc, bt = fill_pools(wl, device)
    q = prefill_queries(wl, qs, device)
    out = torch.empty_like(q)
    qs_d = torch.from_numpy(qs).to(device)
    lens_d = torch.from_numpy(wl.context_lens).to(device)
    flops = prefill_flops(wl.context_lens, qs, wl.n_q_heads, wl.head_dim)
    call = lambda: pk.paged_attention_prefill(q, kc, vc, bt, qs_d, lens_d, wl.scale, out, 512)
    pk.set_option(pk.OPT_PREFILL_PATH, 1)
    ms_mma = timed(call)
    pk.set_option(pk.OPT_PREFILL_PATH, 0)
    ms = timed(call)
    res = {"workload": "16 seqs x 512-token chunk after U[0,3584] cached tokens, Llama-2-7B "
                       "layer (32 heads, D128, fp16, B16)",
           "kernel": "paged_prefill_tc_kernel (tcgen05)",
           "median_us": ms * 1e3, "flops": flops, "tflops": flops / ms / 1e9,
           "peak_tflops": peak, "peak_kind": f"{peak_kind} bf16_tflops (cuBLAS burst)",
           "frac": flops / ms / 1e9 / peak, "kv_bytes": int(2 * wl.context_lens.sum() * wl.row_bytes),
           "warp_mma_kernel": {"median_us": ms_mma * 1e3, "tflops": flops / ms_mma / 1e9,
                               "frac": flops / ms_mma / 1e9 / peak}}
    del kc, vc, q, out
    torch.cuda.empty_cache()
    # a short chunk over a long cached context: 32 items for 152 SMs, whole and
    # with each item's keys split (paged_attention_prefill_split, parts chosen
    # by the library)
    wl3, qs3 = chunked_prefill("chunk128_after16k", "f16", [16384], [128], 32, 32, 128, 16, seed=19)
    kc, vc, bt = fill_pools(wl3, device)
    q = prefill_queries(wl3, qs3, device)
    out = torch.empty_like(q)
    qs_d = torch.from_numpy(qs3).to(device)
    lens_d = torch.from_numpy(wl3.context_lens).to(device)
    ws = pk.prefill_workspace(q)
    whole = timed(lambda: pk.paged_attention_prefill(q, kc, vc, bt, qs_d, lens_d, wl3.scale, out, 128), 20)
    split = timed(lambda: pk.paged_attention_prefill(q, kc, vc, bt, qs_d, lens_d, wl3.scale, out, 128,
                                                     workspace=ws, key_parts=0), 20)
    f3 = prefill_flops(wl3.context_lens, qs3, 32, 128)
    res["chunk128_after16k"] = {"workload": "1 seq, 128-token chunk after 16384 cached tokens, 32 heads, D128, fp16",
                                "whole_us": whole * 1e3, "split_us": split * 1e3,
                                "split_frac": f3 / split / 1e9 / peak}
    assert pk.device_errors() == 0
    del kc, vc, q, out, ws
    torch.cuda.empty_cache()
    if not chunked:
        return res
    # the 2048-token prompt, chunked
    wl2, qs2 = chunked_prefill("prompt2048", "f16", [0], [2048], 32, 32, 128, 16, seed=17)
    kc, vc, bt = fill_pools(wl2, device)
    q = prefill_queries(wl2, qs2, device)
    out = torch.empty_like(q)
    chunking = {}
    for chunk in (2048, 512, 256, 128):
        calls = []
        for c0 in range(0, 2048, chunk):
            rows = q[c0:c0 + chunk]
            o = out[c0:c0 + chunk]
            cqs = torch.tensor([0, chunk], dtype=torch.int32, device=device)
            cl = torch.tensor([c0 + chunk], dtype=torch.int32, device=device)
            calls.append(timed(lambda: pk.paged_attention_prefill(rows, kc, vc, bt, cqs, cl,
                                                                  wl2.scale, o, chunk), 20))
        chunking[str(chunk)] = {"calls": len(calls), "total_us": sum(calls) * 1e3,
                                "max_call_us": max(calls) * 1e3}
    res["prompt2048_chunked"] = chunking
    assert pk.device_errors() == 0
    del kc, vc, q, out
    torch.cuda.empty_cache()
    return res


def compact(fig):
    """The few numbers of a decode figure that the line's tail repeats."""
    return {"frac": round(fig["frac"], 4), "gbs": round(fig["achieved_gbs"], 1),
            "ms": round(fig["decode_ms_back_to_back"], 5),
            "frac_per_call": round(fig["frac_per_call"], 4),
            "frac_l2_flushed": round(fig["frac_l2_flushed"], 4),
            "spread_pct": round(fig["back_to_back_ms_spread"]["range_pct"], 2)}


def run_ours(args, ctx):
    import paged_kv_cache_233_gb300 as pk
    from paged_kv_cache_233_gb300 import build as pk_build
    if ctx.rank == 0:
        pk_build.build()
    ctx.barrier()
    pk_build.build()
    pk.load()
    torch.cuda.set_device(ctx.local_rank)
    device = torch.device("cuda", ctx.local_rank)
    if args.path is not None:
        pk.set_option(pk.OPT_DECODE_PATH, args.path)
    if args.ctas is not None:
        pk.set_option(pk.OPT_CTAS_PER_SM, args.ctas)
    if args.stages is not None:
        pk.set_option(pk.OPT_STAGES, args.stages)
    if args.l2_hints is not None:
        pk.set_option(pk.OPT_L2_HINTS, args.l2_hints)
    wl = workload_for(args.config, ctx.rank)
    if args.seqs is not None:
        wl = subset(wl, range(min(args.seqs, wl.num_seqs)))
    P = PARTITION[args.config] if args.partition is None else args.partition
    step = Step(wl, device, P)
    if args.entry == "shared_prefix":
        step.use_shared_prefix_entry()
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if pk.device_errors():
        raise RuntimeError("device error flags set during warm-up")
    with ClockSampler(torch.cuda.current_device()) as clk:
        total_ms = time_steps(step, args.steps, ctx)
        # the same timed loop again, for the spread of the step time
        repeats = [total_ms / args.steps] + [time_steps(step, args.steps, ctx) / args.steps
                                             for _ in range(args.repeats - 1)]
        # the decode call alone, back to back (the roofline's kernel)
        dec = decode_figures(wl, step.decode, args.gate_reps, args.repeats)
    clocks = clk.summary()
    ms_per_step = total_ms / args.steps
    algo, logical, kv_unique = decode_bytes(wl)
    all_bytes = ctx.sum(algo)
    value = all_bytes / ms_per_step / 1e6                      # GB/s, whole job
    seq_decodes = ctx.sum(wl.num_seqs) / (ms_per_step * 1e-3)
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    e2e_ms, h2d, d2h = time_e2e(step, e2e_steps)
    e2e_ms = ctx.max(e2e_ms)
    peak, peak_kind = measured_peak()
    decode_ms = dec["decode_ms_back_to_back"]
    achieved = algo / decode_ms / 1e6
    result = None
    if ctx.rank == 0:
        result = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ctx.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic",
            "config": workload_config(args.config, wl, P, ctx.world),
            "decode_entry": args.entry,
            "decode_path": {1: "simt", 2: "mma"}.get(pk.last_decode_path()),
            "decode_l2_hints": {0: "auto (K/V stream larger than L2)", 1: "never", 2: "always"}[
                pk.get_option(pk.OPT_L2_HINTS)],
            "step_ms_spread": spread(repeats),
            "seq_decodes_per_s_per_layer": seq_decodes,
            "kv_logical_gbs": ctx.sum(logical) / ms_per_step / 1e6,
            "append_bulk_gbs": append_bytes(wl, step.fill_tokens) / step.fill_ms / 1e6,
            "clocks": clocks,
            "e2e": {"value": all_bytes / e2e_ms / 1e6, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": e2e_steps},
            "gpu_launches": step.launches_per_step * args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": profiled_traffic(args.config, P) if args.seqs is None else None,
                         "peak_kind": f"{peak_kind} hbm_gbs (STREAM-style copy), burst",
                         "kernel": "paged_decode_kernel + its LSE merge (one decode call)",
                         "decode_ms": decode_ms, "algorithmic_bytes_per_launch": algo,
                         "decode_timed_on": f"{args.gate_reps} decode calls back to back, "
                                            f"median of {args.repeats} repeats",
                         "decode_ms_spread": dec["back_to_back_ms_spread"],
                         "decode_ms_per_call": dec["decode_ms_per_call"]},
        }
    del step
    torch.cuda.empty_cache()
    targets = {}
    if ctx.rank == 0 and args.seqs is None:
        targets[args.config] = compact(dec)
    if ctx.rank == 0 and not args.no_cpu_baseline and ctx.world == 1:
        import oracle
        orc = oracle.get()
        wl0, q0, kc, vc = oracle_sample(orc, args.config)
        b, s, n, threads = oracle_rate(orc, wl0, q0, kc, vc, args.cpu_budget)
        b1, s1, n1, _ = oracle_rate(orc, wl0, q0, kc, vc, max(1.0, args.cpu_budget / 4),
                                    threads=1)
        result["cpu_baseline"] = {
            "value": b / s / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} (sequence, kv head) units taken in order, cycling over the "
                      f"{wl0.num_seqs * wl0.n_kv_heads} units of {wl0.name}; {s:.1f} s of "
                      f"fp64 oracle decode on {threads} threads",
            "single_core": {"value": b1 / s1 / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": f"{n1} units, {s1:.1f} s on one thread"}}
        del kc, vc
    if ctx.rank == 0 and not args.no_trace and ctx.world == 1:
        result["trace"] = {f"B{b}_slots{n}": measure_trace(b, device, slots=n)
                           for b in (8, 16, 32) for n in TRACE_SLOTS}
        # a pool of 4,096 token slots instead of 65,536: LIFO preemption by
        # recompute fires (its re-appends run inside the timed steps)
        result["trace"]["B16_slots64_pool4096"] = measure_trace(16, device, slots=64,
                                                                pool_tokens=4096)
        torch.cuda.empty_cache()
        result["cow_copy"] = measure_cow(device)
        result["swap"] = measure_swap(device)
        result["prefill"] = measure_prefill(device)
    if ctx.rank == 0 and not args.no_gates and ctx.world == 1:
        gates = {name: measure_gate(name, args, device)
                 for name in ("gqa8b_prefix", "longctx_splitk", "mha7b") if name != args.config}
        # the long-context workload under the balanced split instead of its stated
        # 512-token partitions (a split the caller may choose; context only)
        gates["longctx_splitk_balanced_split"] = measure_gate("longctx_splitk", args, device,
                                                              partition=-1)
        gates["gqa8b_prefix_shared_prefix_entry"] = measure_shared_prefix(device, args.gate_reps)
        result["gates"] = gates
        for name in ("gqa8b_prefix", "longctx_splitk", "mha7b", "longctx_splitk_balanced_split"):
            if name in gates:
                targets[name] = compact(gates[name])
        sp = gates["gqa8b_prefix_shared_prefix_entry"]
        targets["gqa8b_prefix_shared_prefix_entry"] = {
            k: {"shared": round(v["shared_prefix_entry"]["frac"], 4),
                "plain": round(v["plain_decode"]["frac"], 4)} for k, v in sp.items()}
    if ctx.rank == 0 and "trace" in result:
        targets["trace_decode_gbs"] = {k: round(v["decode_gbs"], 1)
                                       for k, v in result["trace"].items()}
    if ctx.rank == 0 and targets:
        # last key of the line: the decode fractions of the measured HBM peak that
        # the stated targets are about (80% GQA batch 256, 70% long context)
        targets["peak_gbs"] = peak
        result["targets"] = targets
    return result


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="longctx_splitk", choices=sorted(DESCRIPTION))
    ap.add_argument("--seqs", type=int, default=None,
                    help="only the first N sequences of the workload (a smaller case to profile)")
    ap.add_argument("--repeats", type=int, default=5,
                    help="repeats of the timed loops (their spread is reported)")
    ap.add_argument("--partition", type=int, default=None)
    ap.add_argument("--entry", choices=["plain", "shared_prefix"], default="plain",
                    help="decode entry point of the step (shared_prefix: the workload's prefix "
                         "groups through paged_attention_decode_shared_prefix)")
    ap.add_argument("--path", type=int, default=None, help="1 CUDA-core, 2 tensor-core decode")
    ap.add_argument("--ctas", type=int, default=None, help="persistent decode CTAs per SM")
    ap.add_argument("--stages", type=int, default=None, help="decode stage-ring size (2..16)")
    ap.add_argument("--l2-hints", type=int, default=None, choices=(0, 1, 2),
                    help="L2 priorities on the decode's K/V loads: 0 auto (default), 1 never, 2 always")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--gate-reps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--reference-budget", type=float, default=90.0)
    ap.add_argument("--no-gates", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-trace", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="only the chunked-prefill measurement (for profiling its kernel)")
    ap.add_argument("--prefill-reps", type=int, default=50)
    ap.add_argument("--trace-only", type=int, default=None, metavar="BLOCK_SIZE",
                    help="only the continuous-batching trace at this block size (for profiling it)")
    ap.add_argument("--trace-slots", type=int, nargs="+", default=[64],
                    help="slot counts of --trace-only")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.trace_only is not None:
        import paged_kv_cache_233_gb300 as pk
        from paged_kv_cache_233_gb300 import build as pk_build
        pk_build.build()
        pk.load()
        torch.cuda.set_device(0)
        b = args.trace_only
        print(json.dumps({"trace": {f"B{b}_slots{n}": measure_trace(b, torch.device("cuda", 0), slots=n)
                                    for n in args.trace_slots}}), flush=True)
        return
    if args.prefill_only:
        import paged_kv_cache_233_gb300 as pk
        from paged_kv_cache_233_gb300 import build as pk_build
        pk_build.build()
        pk.load()
        torch.cuda.set_device(0)
        print(json.dumps({"prefill": measure_prefill(torch.device("cuda", 0), args.prefill_reps,
                                                     chunked=False)}), flush=True)
        return
    ctx = DistCtx(connect=args.impl == "ours")
    try:
        result = run_reference(args, ctx) if args.impl == "reference" else run_ours(args, ctx)
    finally:
        ctx.close()
    if result is not None:
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
