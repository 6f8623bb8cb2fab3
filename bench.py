"""Benchmark of wt_prepare on the Kimi-K2-shaped MoE layer (384 routed
experts + 1 shared, w1/w3 2048x7168 fused to gate_up 4096x7168, w2
7168x2048, 8 FSDP shards each, FP8 e4m3 128x128 blocks, 8 destination
ranks; 16.96 G params, 33.9 GB BF16 read, 16.96 GB written per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload kimi_k2_moe_layer|llama_dense|llama_dense_tp4|edge_stress|
                              edge_narrow|edge_narrow_1|tiny_dense|offload_8layer|tokens]
                  [--partition replicas|sources] [--sources S] [--shard-local [--fsdp F] [--halo]]
                  [--counters launch|rank] [--images K] [--no-e2e] [--no-cpu-baseline]
                  [--experts E]

Prints one JSON line. `value` is GB/s of BF16 input for the whole job
(all ranks), timed with CUDA events on the launching stream around K
back-to-back steps whose inputs (33.9 GB) are far larger than L2. `e2e`
is the same metric through wt_prepare_offload from pinned host memory,
with the host-to-device copies and the read-back of the step's status
inside the timed region. `--workload offload_8layer` instead times the
8-layer streamed-offload stack (its own JSON line). `--impl reference` times the CPU
oracle on the host cores on a bounded sample of the same workload.
Under torchrun each rank prepares its own layer (weak scaling, no
collective on the data path). With --partition sources the ranks share one
layer and each prepares the outputs that schedule.assign_sources gives it
(strong scaling; --sources 8 at one GPU times rank 0's share). With
--shard-local the ranks instead share one layer as an FSDP group of --fsdp
ranks (default: the world size): rank r holds only shard r of every weight
and prepares the blocks of its own rows with a shard-local plan (strong
scaling; `value` counts the bytes of all ranks); with --halo the halo rows
are exchanged point to point inside every timed step, and `exchange_ms` is
that exchange's share of the step. At one GPU, --shard-local --fsdp 8 times
what one rank of an 8-way group does.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "wt_prepare GB/s (BF16 in) and params/s at 1 B300; % of HBM roofline"
GiB = 1 << 30
SPEC_HBM_GBS = 8000.0
L2_BYTES = 126 * 10**6

# dram__bytes_read.sum + dram__bytes_write.sum of one prep_kernel launch,
# from the ncu capture summarised in profiles/ (16 experts, scaled by the
# blocks processed to the 385-expert layer); valid only for the kernel
# code it was taken on (kernel_sha).
TRAFFIC = {"kernel_sha256": "73bf6d89e7c66e3677cfb3b9597b05c0ec65785b264b71f8e581580bb54995e0",
           "bytes_per_launch": 50029567280, "experts": 385}


_COMMENT_OR_STRING = re.compile(rb'("(?:\\.|[^"\\\n])*")|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(src: bytes) -> bytes:
    """C++ source with its comments removed and whitespace collapsed, so
    that editing a comment does not change what it hashes to."""
    src = _COMMENT_OR_STRING.sub(lambda m: m.group(1) or b" ", src)
    return b" ".join(src.split())


def kernel_sha() -> str:
    """Hash of the preparation kernel's device code: the kernel, the codec,
    the PTX primitives and the device part of plan.h (constants, table
    records, launch arguments; the host-side plan structures after them do
    not reach the kernel), comments and whitespace aside."""
    h = hashlib.sha256()
    for name in ("prep_kernel.cu", "codec.cuh", "ptx.cuh", "plan.h"):
        with open(os.path.join(ROOT, "bf16_fp8_parameter_wt_b300", "csrc", name), "rb") as f:
            src = f.read()
        if name == "plan.h":
            src = src[:src.index(b"// Host-side copy of one param.")]
        h.update(_code_only(src))
    return h.hexdigest()


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def gpu_bus_id(dev) -> str | None:
    """PCI bus id of the device, as nvidia-smi --id takes it."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    try:
        return f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except AttributeError:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if bus_id:
            cmd.insert(1, f"--id={bus_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def mix_2to1_peak(dev, stream, gib: int = 2, reps: int = 5) -> float:
    """DRAM ceiling for the FP8 path's own access mix (2 bytes read : 1
    written): best of `reps` torch adds of two `gib` GiB BF16 tensors into a
    third, GB/s of bytes read + written. The measured copy peak is a 1:1
    mix, which DRAM serves less well, so a streaming kernel with this mix
    can run above it."""
    import torch
    n = gib * GiB // 2
    with torch.cuda.stream(stream):
        a = torch.ones(n, dtype=torch.bfloat16, device=dev)
        b = torch.ones(n, dtype=torch.bfloat16, device=dev)
        c = torch.empty(n, dtype=torch.bfloat16, device=dev)
        best = 0.0
        for _ in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            torch.add(a, b, out=c)
            e1.record(stream)
            stream.synchronize()
            best = max(best, 3 * 2 * n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del a, b, c
    torch.cuda.empty_cache()
    return best


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float, dev) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(world, v: float, dev) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_work(workload, partition: str, world: int, rank: int, fsdp: int = 0,
              halo: bool = False, experts: int = 385, sources: int = 0):
    """What one rank prepares: (workload, Plan keyword arguments, note).
      replicas    : a model of its own (the MoE layer drawn with a per-rank
                    seed; other workloads as they are), the full plan --
                    weak scaling, no exchange;
      sources     : one model shared by every rank (same seeds), and the
                    outputs that assign_sources gives rank `rank` of
                    `sources` source GPUs (default: the world size) --
                    strong scaling, no exchange on the data path;
      shard-local : one model shared by an FSDP group of `fsdp` ranks
                    (default: the world size), sharded `fsdp` ways, and rank
                    r's shard-local plan (halo: boundaries off the 128-row
                    grid, halo rows received from the next ranks) -- strong
                    scaling.
    `workload` is a name, or a workload object shared as it is."""
    from bf16_fp8_parameter_wt_b300.schedule import rank_view
    from workloads import WORKLOADS, kimi_k2_moe_layer
    moe = workload == "kimi_k2_moe_layer"
    if not isinstance(workload, str):
        model = workload
        workload = model.name
        WORKLOADS = {workload: lambda: model}
    if partition == "replicas":
        w = kimi_k2_moe_layer(experts, seed=1003 + rank) if moe else WORKLOADS[workload]()
        return w, {}, f"replicas x{world}" if world > 1 else "single"
    if partition == "sources":
        n = sources or world
        if not 0 <= rank < n:
            raise ValueError(f"rank {rank} has no share among {n} sources")
        w = kimi_k2_moe_layer(experts) if moe else WORKLOADS[workload]()
        sub, mine = rank_view(w, n, rank)
        return sub, {}, f"source {rank} of {n} ({len(mine)} of {len(w.outputs)} outputs by assign_sources)"
    if partition == "shard-local":
        f = fsdp or world
        if not 0 <= rank < f:
            raise ValueError(f"rank {rank} is outside an FSDP group of {f}")
        w = kimi_k2_moe_layer(experts, shards=f) if moe else WORKLOADS[workload]()
        if any(len(p.shard_rows) != f for p in w.params):
            raise ValueError(f"{w.name} has {len(w.params[0].shard_rows)} shards per weight: use that FSDP degree")
        note = f"shard-local rank {rank} of an FSDP group of {f}" + (" with halos" if halo else "")
        return w, {"local_shard": rank, "halo": halo}, note
    raise ValueError(partition)


def rank_groups(w) -> int:
    """Non-empty rank groups of a workload (blocks grouped by the lowest
    rank that holds them): the launches of one step counted per rank."""
    groups = set()
    for o, out in enumerate(w.outputs):
        if out.slices is None or all(sl is None for sl in out.slices):
            groups.add(min(out.dst_ranks))
            continue
        m, n = w.output_shape(o)

        def holds(sl, bi, bj):
            if sl is None:
                return True
            dim, ranges = sl
            b = bi if dim == 0 else bj
            return any(r0 // 128 <= b < -(-(r0 + ln) // 128) for r0, ln in ranges)

        for bi in range(-(-m // 128)):
            for bj in range(-(-n // 128)):
                held = [r for r, sl in zip(out.dst_ranks, out.slices) if holds(sl, bi, bj)]
                groups.add(min(held) if held else 0)
    return len(groups)


def sample_outputs(w, experts: int, target_bytes: int = 700_000_000) -> list:
    """A bounded sample of a workload's outputs: the first `experts` experts
    of an MoE layer, else the outputs in plan order up to about
    target_bytes of BF16 input, skipping any single output larger than that
    (at least one output)."""
    if w.name.startswith("kimi_k2_moe_layer"):
        return list(range(min(len(w.outputs), 2 * experts)))
    out, total = [], 0
    for o in range(len(w.outputs)):
        m, n = w.output_shape(o)
        if 2 * m * n > target_bytes:
            continue
        if out and total + 2 * m * n > target_bytes:
            break
        out.append(o)
        total += 2 * m * n
    return out or [min(range(len(w.outputs)), key=lambda o: w.output_shape(o)[0] * w.output_shape(o)[1])]


def host_cores() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def sample_experts(requested: int) -> int:
    """Experts per CPU-oracle sample: at least one output (gate_up or down)
    per host core, since the oracle parallelises over outputs."""
    return max(requested, -(-host_cores() // 2))


def cpu_baseline(w_full, experts_sample: int, steps: int = 3) -> dict:
    """Time the CPU oracle, as it stands, on a bounded sample of the
    workload's outputs (same shapes, same value recipe): the median of
    `steps` runs."""
    import oracle
    from workloads import make_shards, shards_to_host_u16
    oracle.build()
    outs = sample_outputs(w_full, sample_experts(experts_sample))
    sub = w_full.subset(outs, name=f"{w_full.name}[:{len(outs)} outputs]")
    host = shards_to_host_u16(make_shards(sub, device="cpu"))
    m = oracle.Model(sub)
    cores = host_cores()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        m.prepare(host, nthreads=cores)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    # one thread on the first outputs of the sample (about 50 M params)
    few, n = [], 0
    for i, o in enumerate(outs):
        few.append(i)
        n += sum(sub.params[p].numel for p in sub.outputs[i].parts)
        if n >= 50_000_000:
            break
    one = sub.subset(few, name=f"{sub.name}[:{len(few)}]")
    host1 = shards_to_host_u16(make_shards(one, device="cpu"))
    t0 = time.perf_counter()
    oracle.Model(one).prepare(host1, nthreads=1)
    t1 = time.perf_counter() - t0
    return {"value": round(sub.bytes_read / t / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "params_per_s": round(sub.num_params_total / t, 1),
            "sample": f"{len(outs)} of {len(w_full.outputs)} outputs "
                      f"({sub.num_params_total} params, {sub.bytes_read} B BF16 in), "
                      f"median of {steps} run(s), {t:.2f} s each",
            "single_thread": {"value": round(one.bytes_read / t1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "params_per_s": round(one.num_params_total / t1, 1),
                              "sample": f"first {len(few)} outputs of that sample "
                                        f"({one.num_params_total} params), one run, {t1:.2f} s"}}


def token_cpu_baseline(tokens: int, hidden: int, steps: int = 3) -> dict:
    """Time the CPU oracle's 1 x 128 codec, as it stands, on a seeded
    sample of the batch (same hidden size and value recipe), its tokens
    split over the host cores: the median of `steps` runs."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    import torch
    import oracle
    oracle.build()
    g = torch.Generator().manual_seed(1006)
    z = torch.randn(tokens, hidden, generator=g)
    chi = sum(torch.randn(tokens, hidden, generator=g) ** 2 for _ in range(3))
    bits = (z * 0.02 / torch.sqrt(chi / 3)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    del z, chi
    cores = host_cores()
    chunks = [c for c in np.array_split(np.arange(tokens), cores) if c.size]
    times = []
    with ThreadPoolExecutor(len(chunks)) as ex:
        for _ in range(steps):
            t0 = time.perf_counter()
            list(ex.map(lambda ix: oracle.quantize_tokens(bits[ix[0]:ix[-1] + 1]), chunks))
            times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return {"value": round(2 * tokens * hidden / t / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{tokens} tokens x {hidden} (same recipe), split over {len(chunks)} threads, "
                      f"median of {steps} run(s), {t:.2f} s each"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle timed on the host cores."""
    if rank != 0:
        return
    from workloads import kimi_k2_moe_layer
    w = kimi_k2_moe_layer(args.experts)
    import oracle
    from workloads import make_shards, shards_to_host_u16
    oracle.build()
    n_experts = sample_experts(args.reference_experts)
    sub = w.subset(range(2 * n_experts))
    host = shards_to_host_u16(make_shards(sub, device="cpu"))
    m = oracle.Model(sub)
    cores = host_cores()
    for _ in range(args.warmup):
        m.prepare(host, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        m.prepare(host, nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = sub.bytes_read / dt / 1e9
    sample = (f"each step: {n_experts} of {len(w.outputs) // 2} experts "
              f"({2 * n_experts} outputs for {cores} threads, {sub.num_params_total} params)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded N(0, 0.006) BF16)",
        "params_per_s": round(sub.num_params_total / dt, 1),
        "config": {"workload": w.name, "experts": args.experts, "sample": sample,
                   "parallelism": "replicas" if world > 1 else "single"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="wt", choices=["wt", "reference"])
    ap.add_argument("--experts", type=int, default=385)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-experts", type=int, default=8)
    ap.add_argument("--reference-experts", type=int, default=2,
                    help="experts per reference step (raised to one output per host core)")
    ap.add_argument("--workload", default="kimi_k2_moe_layer",
                    choices=["kimi_k2_moe_layer", "llama_dense", "llama_dense_tp4", "edge_stress",
                             "edge_narrow", "edge_narrow_1", "tiny_dense", "offload_8layer", "tokens"])
    ap.add_argument("--shard-local", action="store_true",
                    help="FSDP group of --fsdp ranks sharing one layer; each prepares its own shard")
    ap.add_argument("--fsdp", type=int, default=0, help="FSDP degree for --shard-local (0: world)")
    ap.add_argument("--halo", action="store_true",
                    help="with --shard-local: shard boundaries off the 128-row grid, halo rows exchanged")
    ap.add_argument("--partition", default="replicas", choices=["replicas", "sources"],
                    help="under torchrun: a layer per rank (replicas) or one layer split over "
                         "the ranks by assign_sources (sources)")
    ap.add_argument("--sources", type=int, default=0,
                    help="with --partition sources: number of source GPUs (0: world size); "
                         "at one GPU, --sources 8 times rank 0's share")
    ap.add_argument("--counters", choices=["launch", "rank"], default=None,
                    help="time the step with per-rank completion counters")
    ap.add_argument("--tokens", type=int, default=131072)
    ap.add_argument("--cpu-tokens", type=int, default=32768,
                    help="tokens of the sample the CPU oracle is timed on (--workload tokens)")
    ap.add_argument("--hidden", type=int, default=7168)
    ap.add_argument("--images", type=int, default=2)
    ap.add_argument("--stack-steps", type=int, default=2)
    ap.add_argument("--stack-warmup", type=int, default=1)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup() if args.impl == "wt" else (
        int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.workload == "offload_8layer":
        run_offload_stack(args, world, rank, local)
        return
    if args.workload == "tokens":
        run_tokens(args, world, rank, local)
        return

    import torch
    import bf16_fp8_parameter_wt_b300 as wt
    from bf16_fp8_parameter_wt_b300 import build as wt_build
    from workloads import WORKLOADS, kimi_k2_moe_layer, make_shards

    wt_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    partition = "shard-local" if args.shard_local else args.partition
    if args.halo and partition != "shard-local":
        ap.error("--halo needs --shard-local")
    if partition != "replicas" and args.workload in ("offload_8layer", "tokens"):
        ap.error(f"--partition {partition} prepares a plan workload")
    fsdp = (args.fsdp or world) if partition == "shard-local" else 0
    try:
        w, plan_kw, parallelism = rank_work(args.workload, partition, world, rank, fsdp=fsdp,
                                            halo=args.halo, experts=args.experts, sources=args.sources)
    except ValueError as e:
        ap.error(str(e))
    plan = wt.Plan(w, device=local, **plan_kw)
    shards = make_shards(w, device=dev)
    halo_bytes = 0
    exchange = None            # the per-step halo exchange under torchrun
    if partition == "shard-local":
        # this rank keeps its own shard of every weight, plus the halo rows
        # its plan reads from other shards: received from their ranks into
        # fixed buffers under torchrun (every timed step exchanges them
        # again), cut from the locally drawn copy at one GPU
        need = {(i, k): plan.shard_rows_read(i, k) for i, per in enumerate(shards)
                for k in range(len(per)) if k != rank}
        if world > 1 and args.halo:
            if fsdp != world:
                ap.error("exchanging halos needs --fsdp equal to the world size")
            from bf16_fp8_parameter_wt_b300.schedule import exchange_halos, halo_buffers, halo_transfers
            transfers = halo_transfers(w, fsdp)
            got = halo_buffers(w, transfers, rank, dev)
            own = [per[rank] for per in shards]
            barrier(world)                     # a collective before the first point-to-point batch

            def exchange():
                exchange_halos(w, transfers, rank, own, out=got)

            exchange()
        else:
            got = {key: shards[key[0]][key[1]][:n].clone() for key, n in need.items() if n}
        shards = [[s if k == rank else got.get((i, k), s.new_empty(0)) for k, s in enumerate(per)]
                  for i, per in enumerate(shards)]
        halo_bytes = sum(t.numel() * 2 for t in got.values())
        torch.cuda.empty_cache()
    flat = [s for per in shards for s in per]
    shard_ptrs = [s.data_ptr() if s.numel() else 0 for s in flat]
    st = plan.stats
    pools = [torch.empty(max(1, plan.pool_bytes(r)), dtype=torch.uint8, device=dev)
             for r in range(w.num_ranks)]
    pool_ptrs = [p.data_ptr() for p in pools]
    shard_ptrs, pool_ptrs = plan.bind(shard_ptrs, pool_ptrs)
    counters = None
    if args.counters:
        counters = torch.zeros(w.num_ranks, dtype=torch.int32, device=dev)
        plan.set_counters(counters.data_ptr(),
                          wt.WT_COUNT_PER_RANK if args.counters == "rank" else wt.WT_COUNT_PER_LAUNCH)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream

    # the first step stages the pointers: one tensor map per shard is
    # encoded on the host and uploaded with the destination addresses
    t_first = time.perf_counter()
    plan.prepare(shard_ptrs, pool_ptrs, sp)
    first_step_host_ms = (time.perf_counter() - t_first) * 1e3
    with torch.cuda.stream(stream):
        for _ in range(args.warmup - 1):
            if exchange:
                exchange()
            plan.prepare(shard_ptrs, pool_ptrs, sp)
    stream.synchronize()

    bus = gpu_bus_id(dev)
    # a step is [halo exchange (torchrun, --halo)] + wt_prepare; the launch's
    # own time runs from `mids` to `ends`
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if exchange else starts
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(bus)
    time.sleep(0.3)
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            starts[i].record(stream)
            if exchange:
                exchange()             # NCCL point-to-point; its completion is ordered on `stream`
                mids[i].record(stream)
            plan.prepare(shard_ptrs, pool_ptrs, sp)
            ends[i].record(stream)
    stream.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    clk = clocks.stop()
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(mids, ends)]
    exchange_ms = (round(statistics.mean(s.elapsed_time(m) for s, m in zip(starts, mids)), 4)
                   if exchange else None)
    total_ms = starts[0].elapsed_time(ends[-1])
    total_ms = max_over_ranks(world, total_ms, dev)
    ms_per_step = total_ms / args.steps
    # the units every rank processed (replicas: each a whole layer; shard-local:
    # each its own share of one layer)
    job_bytes = sum_over_ranks(world, st["bytes_read"], dev)
    job_params = sum_over_ranks(world, st["num_params_total"], dev)
    value = job_bytes / (ms_per_step * 1e-3) / 1e9
    params_per_s = job_params / (ms_per_step * 1e-3)
    avg_launch_s = statistics.mean(per_launch_ms) * 1e-3
    alg_bytes = st["bytes_read"] + st["bytes_written"]
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    achieved = alg_bytes / avg_launch_s / 1e9
    traffic = (TRAFFIC["bytes_per_launch"]
               if TRAFFIC["kernel_sha256"] == kernel_sha() and args.workload == "kimi_k2_moe_layer"
               and TRAFFIC["experts"] == args.experts and partition == "replicas" else None)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak if peak else 6400.0, "unit": "GB/s",
                "frac": round(achieved / (peak if peak else 6400.0), 4),
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak else "fallback",
                "frac_of_8TBs_spec": round(achieved / SPEC_HBM_GBS, 4),
                "traffic": traffic, "algorithmic_bytes_per_launch": alg_bytes,
                "kernel": "prep_kernel", "launch_ms_median": round(statistics.median(per_launch_ms), 4),
                "launch_ms_min": round(min(per_launch_ms), 4)}
    if 4 * st["bytes_written"] <= 3 * st["bytes_read"]:
        # the FP8 path reads two bytes per byte it writes: its own ceiling,
        # measured live next to the copy peak
        mix = mix_2to1_peak(dev, stream)
        roofline["mix_2to1_peak"] = round(mix, 1)
        roofline["frac_of_mix_2to1_peak"] = round(achieved / mix, 4)
    if roofline["frac"] > 1.0:
        roofline["note"] = ("frac > 1: the measured peak is a 1:1 read:write copy; this kernel's "
                            "read:write mix is served faster by DRAM (see mix_2to1_peak)")

    graph_us = None
    if st["bytes_read"] <= L2_BYTES:
        # an L2-resident step is a latency figure: replay it from a CUDA graph
        # so that the Python call around it is not timed, and 20 steps in one
        # graph so that the host is not timed either
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(20):
                plan.prepare(shard_ptrs, pool_ptrs, sp)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):          # replay() launches on the current stream
            for _ in range(3):
                graph.replay()
            g0.record(stream)
            graph.replay()
            g1.record(stream)
            stream.synchronize()
        plan.check(sp)
        graph_us = round(g0.elapsed_time(g1) * 1e3 / 20, 2)

    e2e = None
    if partition == "shard-local":
        e2e = {"value": None, "reason": "shard-local plans do not stage offloaded shards"}
    elif not args.no_e2e:
        del pools
        torch.cuda.empty_cache()
        e2e = measure_e2e(w, shards, args, dev, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on a sample of the whole workload, whichever share of it
        # the partition gives this rank
        del shards, flat
        torch.cuda.empty_cache()
        cpu = cpu_baseline(w, args.cpu_experts)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak" if partition == "replicas" else "strong",
        "vs_baseline": None, "dtype": "f32",
        "data": f"synthetic (seeded {w.values.dist}, sigma {w.values.sigma}, BF16, generated on device)",
        "params_per_s": round(params_per_s, 1),
        "hbm_frac_of_8TBs_spec": round(value * (alg_bytes / st["bytes_read"]) / SPEC_HBM_GBS, 4),
        "config": {"workload": w.name, "params_per_rank": st["num_params_total"],
                   "bytes_read_per_rank": st["bytes_read"], "bytes_written_per_rank": st["bytes_written"],
                   "io": "BF16 in; e4m3 codes + fp32 128x128 scales out (BF16 pass-through where set)",
                   "l2": (f"inputs ({st['bytes_read'] / 1e9:.1f} GB) larger than the 126 MB L2, no flush"
                          if st["bytes_read"] > L2_BYTES else
                          "inputs smaller than L2: L2-resident, a latency figure"),
                   "halo_bytes_per_rank": halo_bytes if partition == "shard-local" else None,
                   "parallelism": parallelism},
        "exchange_ms": exchange_ms,
        "roofline": roofline, "graph_replay_us": graph_us,
        "first_step_host_ms": round(first_step_host_ms, 2), "shards": st["num_slots"],
        "completion_counters": args.counters,
        "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
        # the preparation kernel, plus the count kernel when counting per
        # launch; per rank, one of each per non-empty rank group
        "gpu_launches": args.steps * (2 if args.counters == "launch" else
                                      2 * rank_groups(w) if args.counters == "rank" else 1),
        "wall_s_timed": round(t_wall, 4),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_tokens(args, world, rank, local):
    """The 1 x 128 activation codec (wt_quantize_tokens) on a dispatch-shaped
    batch: --tokens x --hidden BF16 (Student-t(3) x 0.02), codes and scales
    written to device buffers, stages handed out from a ticket counter; the
    large default batch (1.9 GB) is larger than L2, a 128-token batch gives
    the per-dispatch latency."""
    import torch
    import bf16_fp8_parameter_wt_b300 as wt
    from bf16_fp8_parameter_wt_b300 import build as wt_build
    wt_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    T, H = args.tokens, args.hidden
    G = -(-H // 128)
    g = torch.Generator(device=dev).manual_seed(1006 + rank)
    z = torch.randn(T, H, generator=g, device=dev)
    chi = sum(torch.randn(T, H, generator=g, device=dev) ** 2 for _ in range(3))
    x = (z.mul_(0.02).div_(chi.div_(3).sqrt_())).to(torch.bfloat16)
    del z, chi
    codes = torch.empty(T, H, dtype=torch.uint8, device=dev)
    scales = torch.empty(T, G, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    ticket = torch.zeros(2, dtype=torch.int32, device=dev)   # stage counter of the calls on `stream`

    def step():
        wt.wt_quantize_tokens(x.data_ptr(), T, H, H, codes.data_ptr(), scales.data_ptr(),
                              stream.cuda_stream, ticket.data_ptr())

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    small = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(gpu_bus_id(dev))
    time.sleep(0.3)
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    stream.synchronize()
    clk = clocks.stop()
    wt.wt_tokens_check(stream.cuda_stream)       # no wait of the timed launches gave up
    per = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = max_over_ranks(world, starts[0].elapsed_time(ends[-1]) / args.steps, dev)
    # one dispatch-sized call (128 tokens), latency only: `reps` calls
    # captured in one CUDA graph and replayed at once, so that the time is
    # the GPU's per call (kernel and launch gap), not the host's rate of
    # submitting graph launches
    reps = 20
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(reps):
            wt.wt_quantize_tokens(x.data_ptr(), 128, H, H, codes.data_ptr(), scales.data_ptr(),
                                  stream.cuda_stream, ticket.data_ptr())
    with torch.cuda.stream(stream):              # replay() launches on the current stream
        for _ in range(3):
            graph.replay()
        small[0].record(stream)
        graph.replay()
        small[1].record(stream)
        stream.synchronize()
    wt.wt_tokens_check(stream.cuda_stream)
    bytes_in = 2 * T * H
    alg = bytes_in + T * H + 4 * T * G
    peak = measured_peaks().get("hbm_gbs") or 6400.0
    achieved = alg / (statistics.mean(per) * 1e-3) / 1e9
    del graph, x, codes, scales
    torch.cuda.empty_cache()
    mix = mix_2to1_peak(dev, stream)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = token_cpu_baseline(min(args.cpu_tokens, T), H)
    line = {
        "metric": "wt_quantize_tokens GB/s (BF16 in), 1x128 e4m3 activation codec",
        "value": round(world * bytes_in / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Student-t(3) x 0.02 BF16, generated on device)",
        "config": {"workload": f"tokens_{T}x{H}", "tokens": T, "hidden": H,
                   "l2": "inputs larger than the 126 MB L2, no flush" if bytes_in > L2_BYTES else
                         "inputs smaller than L2"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "frac_of_8TBs_spec": round(achieved / SPEC_HBM_GBS, 4),
                     "algorithmic_bytes_per_launch": alg, "kernel": "token_ring_kernel",
                     "launch_ms_median": round(statistics.median(per), 4),
                     "mix_2to1_peak": round(mix, 1), "frac_of_mix_2to1_peak": round(achieved / mix, 4)},
        "dispatch_128_tokens_us": round(small[0].elapsed_time(small[1]) * 1e3 / reps, 2),
        "cpu_baseline": cpu, "clocks": clk, "gpu_launches": args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def pinned_budget(world: int) -> float:
    """Pinned host bytes one rank may take for the end-to-end leg: 40 % of
    the host's memory shared by the ranks on it (no limit if it cannot be
    read)."""
    try:
        import psutil
        return 0.4 * psutil.virtual_memory().total / max(1, world)
    except Exception:
        return float("inf")


def e2e_subset(w, shards, host_bytes: int, budget: float):
    """Every rank pins its own host image for the end-to-end leg: when the
    MoE layer's image is over the rank's budget, take the first experts
    that fit (the step is bound by the host-to-device link, so its GB/s
    does not depend on how many experts there are). Returns (workload,
    shards, sample note or None)."""
    if host_bytes <= budget or not w.name.startswith("kimi_k2_moe_layer"):
        return w, shards, None
    per_expert = host_bytes / (len(w.outputs) // 2)
    experts = max(1, int(budget // per_expert))
    sub = w.subset(range(2 * experts), name=f"{w.name}[:{experts} experts]")
    return sub, shards[:3 * experts], f"first {experts} experts per rank"


def pinned_image(plan, shards):
    """The packed pinned host image that wt_prepare_offload reads."""
    import torch
    host = torch.empty(plan.stats["host_bytes"], dtype=torch.uint8, pin_memory=True)
    for p, per in enumerate(shards):
        for k, s in enumerate(per):
            off = plan.shard_host_offset(p, k)
            n = s.numel() * 2
            host[off:off + n].copy_(s.reshape(-1).view(torch.uint8))
    return host


def h2d_peak(host, dev, stream, reps: int = 3) -> float:
    """Best of `reps` plain pinned 2 GiB host-to-device copies (GB/s): the
    bound of the offload path."""
    import torch
    n = min(2 * GiB, host.numel())
    buf = torch.empty(n, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            buf.copy_(host[:n], non_blocking=True)
        e1.record(stream)
        stream.synchronize()
        best = max(best, n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    return best


def measure_e2e(w, shards, args, dev, world):
    """The same step through the public API from pinned host memory: each
    step is wt_prepare_offload (2 GiB chunks copied host-to-device on one
    stream while the previous chunk is prepared on another) followed by
    wt_plan_check, which waits for the step and reads its 4-byte status
    back to the host. The destination pools stay on the device: they stand
    in for the remote inference memory the prepared bytes are written to."""
    import torch
    import bf16_fp8_parameter_wt_b300 as wt
    plan = wt.Plan(w, device=dev.index, offload_chunk_bytes=2 * GiB)
    st = plan.stats
    w, shards, sample = e2e_subset(w, shards, st["host_bytes"], pinned_budget(world))
    if sample:
        plan.close()
        plan = wt.Plan(w, device=dev.index, offload_chunk_bytes=2 * GiB)
        st = plan.stats
        sample += f" (pinned image {st['host_bytes'] / 1e9:.1f} GB)"
    host = pinned_image(plan, shards)
    pools = [torch.empty(max(1, plan.pool_bytes(r)), dtype=torch.uint8, device=dev)
             for r in range(w.num_ranks)]
    pool_ptrs = [p.data_ptr() for p in pools]
    copy_s, comp_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def step():
        plan.prepare_offload(host.data_ptr(), pool_ptrs, copy_s.cuda_stream, comp_s.cuda_stream)
        plan.check(comp_s.cuda_stream)

    step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        step()
    dt = (time.perf_counter() - t0) / args.e2e_steps
    dt = max_over_ranks(world, dt, dev)
    peak = h2d_peak(host, dev, copy_s)
    plan.close()
    return {"value": round(world * st["bytes_read"] / dt / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": st["host_bytes"], "d2h_bytes_per_step": 4,
            "ms_per_step": round(dt * 1e3, 2), "chunks": st["num_chunks"],
            "h2d_peak_gbs": round(peak, 2),
            "overlap_efficiency": round(st["host_bytes"] / (peak * 1e9) / dt, 4),
            "api": "wt_prepare_offload + wt_plan_check (status read)",
            "workload": w.name, "sample": sample}


def run_offload_stack(args, world, rank, local):
    """The streamed-offload stack: 8 layers, each the MoE layer plus q/k/v/o
    7168x7168 projections (qkv fused), held as BF16 shards in pinned host
    memory and prepared through wt_prepare_offload into one set of pools
    reused by every layer. The host holds `--images` distinct layer images
    (seeded draws) that the 8 layers cycle through, so the pinned footprint
    fits the host; host-to-device traffic is that of 8 distinct layers."""
    import torch
    import bf16_fp8_parameter_wt_b300 as wt
    from bf16_fp8_parameter_wt_b300 import build as wt_build
    from workloads import make_shards, offload_layer

    wt_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = offload_layer(args.experts, seed=1005 + 100 * rank)
    plan = wt.Plan(w, device=local, offload_chunk_bytes=2 * GiB)
    st = plan.stats
    # the ranks on one host share its memory: fewer distinct images (the
    # host-to-device traffic stays that of 8 layers), never none
    budget = pinned_budget(world)
    fit = args.images if budget == float("inf") else int(budget // max(1, st["host_bytes"]))
    n_images = max(1, min(args.images, fit))
    images = []
    for i in range(n_images):
        wi = offload_layer(args.experts, seed=1005 + 100 * rank + i)
        shards = make_shards(wi, device=dev)
        images.append(pinned_image(plan, shards))
        del shards
        torch.cuda.empty_cache()
    pools = [torch.empty(max(1, plan.pool_bytes(r)), dtype=torch.uint8, device=dev)
             for r in range(w.num_ranks)]
    pool_ptrs = [p.data_ptr() for p in pools]
    copy_s, comp_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    layers = 8

    def step():
        for layer in range(layers):
            plan.prepare_offload(images[layer % len(images)].data_ptr(), pool_ptrs,
                                 copy_s.cuda_stream, comp_s.cuda_stream)
        plan.check(comp_s.cuda_stream)

    for _ in range(args.stack_warmup):
        step()
    barrier(world)
    clocks = ClockSampler(gpu_bus_id(dev))
    time.sleep(0.3)
    t0 = time.perf_counter()
    for _ in range(args.stack_steps):
        step()
    dt = (time.perf_counter() - t0) / args.stack_steps
    clk = clocks.stop()
    dt = max_over_ranks(world, dt, dev)
    peak = h2d_peak(images[0], dev, copy_s)
    plan.close()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_experts)
    host_bytes = layers * st["host_bytes"]
    value = world * layers * st["bytes_read"] / dt / 1e9
    line = {
        "metric": "wt_prepare_offload GB/s (BF16 host in), 8-layer streamed offload",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.stack_steps,
        "warmup": args.stack_warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0, 0.006) BF16, pinned host images)",
        "params_per_s": round(world * layers * st["num_params_total"] / dt, 1),
        "config": {"workload": f"offload_stack_8x{w.name}", "layers": layers,
                   "host_images": n_images, "chunk_bytes": 2 * GiB, "chunks_per_layer": st["num_chunks"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": host_bytes,
                "d2h_bytes_per_step": 4},
        "h2d_peak_gbs": round(peak, 2),
        "overlap_efficiency": round(host_bytes / (peak * 1e9) / dt, 4),
        "cpu_baseline": cpu, "clocks": clk,
        # one preparation launch per chunk of every layer
        "gpu_launches": args.stack_steps * layers * st["num_chunks"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
