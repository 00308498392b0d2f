"""Benchmark of the Clef JointSchemaHead forward pass on GB300.

One step = one whole head forward (pooling, option queries, memory K/V projection,
routing layers, fields, joint layers, scorer, softmax) over one batch of the
workload, inputs resident in HBM.  Default workload: 8 records of 16384 memory rows
(hidden 4096) with a 16-question schema, the batch the headline metric is quoted on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead,
on a bounded sample of the same workload (the only other place this file runs the
oracle is the ``cpu_baseline`` leg).  Under torchrun the job holds one batch of
N x 8 records of the same shape; ``shard_records`` gives every rank its own 8 (weak
scaling: records are independent, so there is no collective on the data path) and
each rank draws and uploads only its own records.  After the timed region the
per-rank outputs are gathered once through ``ShardedRunner`` and checked.
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

NCPU = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(NCPU))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "head records/s & memory tokens/s (16K ctx, batch 8); % of BF16 TC / HBM roofline"
WORKLOAD = "batch8_l16k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dram__bytes_read.sum + dram__bytes_write.sum of one full K/V-projection launch of this
# workload: an ncu capture of the same kernel on the first 2 records, scaled to 8 records
# (set to None whenever the kernel changes until it is captured again).
KV_GEMM_TRAFFIC_BYTES = 2.288e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {}
        for k in FALLBACK_PEAKS:
            v = d.get(k)
            if isinstance(v, dict):
                v = v.get("value")
            out[k] = float(v) if v is not None else None
        if all(v is not None for v in out.values()):
            return out, "measured"
    except (OSError, ValueError, TypeError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu, self.rows, self.proc = str(gpu_index), [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", self.gpu, "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kv_gemm_flops(T, H, D, n_route):
    """Algorithmic flops of the memory K/V projection: 2 * H * (2 * n_route * D) per real token."""
    return 2.0 * H * (2 * n_route * D) * T


def attn_bytes(T, D):
    """Algorithmic HBM bytes of one routing layer's attention: K and V rows of every real token, bf16."""
    return 2.0 * 2 * D * T


def pool_bytes(bt):
    """Algorithmic HBM bytes of span pooling: every span row read once (hidden, plus the
    lexical row for option spans), the global row, and the pooled outputs written."""
    H = bt.H
    q_rows = int((bt.q_span[:, 1] - bt.q_span[:, 0]).sum())
    o_rows = int((bt.o_span[:, 1] - bt.o_span[:, 0]).sum())
    read = (q_rows + 2 * o_rows + bt.B) * H * 2
    write = (bt.Q * (4 + 2 + 0) + bt.O * (2 + 2 + 4) + bt.B * 4) * H + bt.O * H * 2  # fp32 + bf16 copies
    return float(read + write)


def oracle_one_record(w, shape, bt, b):
    import oracle
    t0 = time.perf_counter()
    oracle.head_forward(w, shape.heads, shape.n_route, shape.n_joint, bt.record_hidden, bt.lengths, bt.q_rec,
                        bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span, bt.token_ids, bt.lexical, records=[b])
    return time.perf_counter() - t0


def local_batch(bt_g, sb):
    """The records of one shard as a batch of their own: tables re-indexed from zero,
    padded to the shard's longest record, hidden rows drawn for these records only."""
    recs = sb.records
    Lp = int(sb.lengths.max())
    hid = np.stack([bt_g.record_hidden(int(b))[:Lp] for b in recs])
    return dataclasses.replace(bt_g, B=len(recs), Lpad=Lp, lengths=sb.lengths, q_rec=sb.q_rec, q_type=sb.q_type,
                               q_span=sb.q_span, q_opt_off=sb.q_opt_off, o_span=sb.o_span,
                               token_ids=np.ascontiguousarray(bt_g.token_ids[recs, :Lp]), hidden=hid)


def run_reference(args, spec, shape):
    """The oracle as it stands, timed on the host cores: one step = one record."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    bt = synth.make_batch(spec, seed=1, with_hidden=False)
    w = synth.make_weights(shape, seed=0)
    budget = float(os.environ.get("CLEF_REFERENCE_BUDGET_S", "150"))
    t_start = time.perf_counter()
    for i in range(args.warmup):  # untimed, like the GPU arm's warm-up steps
        oracle_one_record(w, shape, bt, i % bt.B)
    times = []
    for i in range(args.steps):
        times.append(oracle_one_record(w, shape, bt, i % bt.B))
        if time.perf_counter() - t_start > budget:
            break
    step_s = sum(times) / len(times)
    tokens = float(bt.lengths.mean())
    value = 1.0 / step_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "records/s", "n_gpus": args.gpus,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators, random-init head weights)",
        "config": {"workload": spec.name, "records_per_step": 1, "hidden": shape.H, "memory_rows": int(tokens)},
        "memory_tokens_per_s": tokens / step_s,
        "cpu_baseline": {"value": value, "unit": "records/s", "cores": NCPU, "kind": "oracle",
                         "sample": f"one record of {spec.name} per step ({int(tokens)} memory rows), fp64 NumPy"},
        "e2e": {"value": value, "unit": "records/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--records", type=int, default=0, help="use only the first N records (profiling cases)")
    ap.add_argument("--stream-chunk", type=int, default=64,
                    help="rows per chunk of the streaming-ingestion leg (0: skip the leg)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    spec = synth.workload_spec(args.workload)
    if args.records:
        spec = dataclasses.replace(spec, B=args.records,
                                   lengths=None if spec.lengths is None else list(spec.lengths)[:args.records])
    shape = synth.HeadShape(H=spec.H)
    if args.impl == "reference":
        run_reference(args, spec, shape)
        return

    import torch
    import torch.distributed as dist

    from structured_decision_model_gb300 import binding as B
    from structured_decision_model_gb300.build import build_library
    from structured_decision_model_gb300.head import ClefHead, to_device_bf16
    from structured_decision_model_gb300.sharding import ShardedRunner, shard_records, sub_batch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    build_library()
    B.load()

    # one batch of world x B records; this rank's shard (B records, weak scaling) is
    # picked by the same row-balanced split ShardedRunner uses
    spec_g = spec if world == 1 else dataclasses.replace(
        spec, B=spec.B * world, lengths=None if spec.lengths is None else list(spec.lengths) * world)
    bt_g = synth.make_batch(spec_g, seed=1, with_hidden=(world == 1))
    tables = (bt_g.lengths, bt_g.q_rec, bt_g.q_type, bt_g.q_span, bt_g.q_opt_off, bt_g.o_span)
    shards = shard_records(bt_g.lengths, world)
    sb = sub_batch(shards[rank], *tables)
    bt = bt_g if world == 1 else local_batch(bt_g, sb)
    w = synth.make_weights(shape, seed=0)
    head = ClefHead(w, shape.H, shape.D, shape.heads, shape.F, shape.n_route, shape.n_joint, shape.vocab, device=dev)
    schema = B.Schema(bt.B, bt.Lpad, bt.H, bt.lengths, bt.q_rec, bt.q_type, bt.q_span, bt.q_opt_off, bt.o_span)
    hidden_host = torch.from_numpy(bt.hidden.view(np.int16)).view(torch.bfloat16)
    hidden = hidden_host.to(dev)
    ids_host = torch.from_numpy(bt.token_ids)
    ids = ids_host.to(dev)
    lexical = torch.empty((shape.vocab, shape.H), dtype=torch.bfloat16, device=dev)
    lexical.normal_(0.0, 0.02, generator=torch.Generator(device=dev).manual_seed(0))
    used = bt.lexical_ids()
    lexical[torch.from_numpy(used.astype(np.int64)).to(dev)] = to_device_bf16(bt.lexical[used], dev)
    out = head.alloc_outputs(schema)
    stream = torch.cuda.current_stream()

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
        for e in evs:
            e.record(stream)  # creates the event handle
        return evs

    for _ in range(args.warmup):
        head.forward(schema, hidden, ids, lexical, out=out)
    torch.cuda.synchronize()
    if head.device_status() != 0:
        raise RuntimeError("device status after warm-up is not OK")

    K = args.steps
    ev_sets = [new_events() for _ in range(K)]
    dbgs = []
    for evs in ev_sets:
        d = B.ClefDebugOutputs()
        for i, e in enumerate(evs):
            d.events[i] = e.cuda_event
        dbgs.append(d)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = B.clef_kernel_launches()
    with ClockSampler(dev.index) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(K):
            head.forward(schema, hidden, ids, lexical, out=out, debug=dbgs[i])
        stop.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    launches = B.clef_kernel_launches() - launches0
    status = head.device_status()
    if status != 0:
        raise RuntimeError(f"device status {B.STATUS.get(status, status)}")
    ms = start.elapsed_time(stop) / K
    kv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev_sets)
    att_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev_sets)
    pool_ms = statistics.mean(e[4].elapsed_time(e[5]) for e in ev_sets)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # end to end through the C ABI: every step copies its inputs from pinned host memory
    # and reads its results back.  Two device input buffers let the copy of step i + 1
    # (on a copy stream) overlap the head of step i.
    e2e_value = None
    h2d = hidden_host.numel() * 2 + ids_host.numel() * 4
    d2h = schema.O * 4 * 2 + schema.Q * 4 * 3
    if args.e2e_steps > 0:
        hid_pin = hidden_host.pin_memory()
        ids_pin = ids_host.pin_memory()
        res_pin = [torch.empty(n, dtype=dt).pin_memory() for n, dt in
                   ((schema.O, torch.float32), (schema.O, torch.float32), (schema.Q, torch.float32),
                    (schema.Q, torch.float32), (schema.Q, torch.int32))]
        outs = (out.logits, out.probs, out.q_value, out.q_conf, out.q_argmax)
        in_bufs = [(hidden, ids), (torch.empty_like(hidden), torch.empty_like(ids))]
        copy_stream = torch.cuda.Stream(device=dev)
        ready = [torch.cuda.Event(), torch.cuda.Event()]
        free = [torch.cuda.Event(), torch.cuda.Event()]

        def issue_copy(i):
            k = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(free[k])
                in_bufs[k][0].copy_(hid_pin, non_blocking=True)
                in_bufs[k][1].copy_(ids_pin, non_blocking=True)
                ready[k].record(copy_stream)

        def run_e2e(n):
            issue_copy(0)
            for i in range(n):
                k = i % 2
                if i + 1 < n:
                    issue_copy(i + 1)
                stream.wait_event(ready[k])
                head.forward(schema, in_bufs[k][0], in_bufs[k][1], lexical, out=out)
                free[k].record(stream)
                for dst, src in zip(res_pin, outs):
                    dst.copy_(src, non_blocking=True)

        run_e2e(2)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        run_e2e(args.e2e_steps)
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
        if world > 1:
            t = torch.tensor([e2e_ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_ms = float(t.item())
        e2e_value = world * bt.B / (e2e_ms / 1e3)

    # streaming ingestion: memory rows arrive in chunks (records interleaved); the head
    # finishes after the last chunk.  finish_ms is the latency from the last chunk to the
    # answers, to compare with a whole forward's ms_per_step.
    stream_info = None
    if args.stream_chunk > 0:
        C = args.stream_chunk
        chunks = [(b, r0, min(C, int(bt.lengths[b]) - r0)) for r0 in range(0, int(bt.lengths.max()), C)
                  for b in range(bt.B) if r0 < bt.lengths[b]]

        def stream_pass(ev=None):
            head.stream_begin(schema)
            for (b, r0, n) in chunks:
                head.stream_rows(schema, hidden, b, r0, n)
            if ev is not None:
                ev.record(stream)
            head.stream_finish(schema, hidden, ids, lexical, out=out)

        stream_pass()
        torch.cuda.synchronize()
        s0, s1, s2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        t_host = time.perf_counter()
        s0.record(stream)
        stream_pass(s1)
        s2.record(stream)
        torch.cuda.synchronize()
        t_host = time.perf_counter() - t_host
        if head.device_status() != 0:
            raise RuntimeError("device status after the streaming leg is not OK")
        stream_info = {"chunk_rows": C, "chunks": len(chunks), "finish_ms": s1.elapsed_time(s2),
                       "ingest_ms": s0.elapsed_time(s1), "host_us_per_chunk": t_host * 1e6 / len(chunks),
                       "forward_ms": ms}

    # the gather of the sharded runner: every rank's outputs, once, after the timed
    # region; checked against this rank's own outputs (a few KB per rank)
    sharded = None
    if world > 1:
        mine = {"logits": out.logits.cpu().numpy(), "probs": out.probs.cpu().numpy(),
                "value": out.q_value.cpu().numpy(), "conf": out.q_conf.cpu().numpy(),
                "argmax": out.q_argmax.cpu().numpy()}
        full = ShardedRunner(lambda _sb: mine).forward(*tables)
        ok = bool(np.array_equal(full["logits"][sb.o_index], mine["logits"]) and np.isfinite(full["logits"]).all())
        sharded = {"records_total": int(bt_g.B), "records_per_rank": [len(x) for x in shards], "gather_ok": ok}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        recs = list(range(min(3, bt.B)))
        dts = [oracle_one_record(w, shape, bt, b) for b in recs]
        dt = statistics.median(dts)
        cpu = {"value": 1.0 / dt, "unit": "records/s", "cores": NCPU, "kind": "oracle",
               "sample": f"records {recs} of the batch ({int(bt.lengths[0])} memory rows, "
                         f"{int((bt.q_rec == 0).sum())} questions each), one record per timing, median of "
                         f"{len(recs)}; the oracle is fp64 NumPy (slower than an fp32 program would be), "
                         f"{sum(dts):.1f} s in total"}

    if rank == 0:
        peaks, peak_src = load_peaks()
        T = bt.T
        kv_flops = kv_gemm_flops(T, shape.H, shape.D, shape.n_route)
        kv_tf = kv_flops / (kv_ms * 1e-3) / 1e12
        att_gbs = attn_bytes(T, shape.D) / (att_ms * 1e-3) / 1e9
        pool_gbs = pool_bytes(bt) / (pool_ms * 1e-3) / 1e9
        records_s = world * bt.B / (ms / 1e3)
        line = {
            "metric": METRIC, "value": records_s, "unit": "records/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generators, random-init head weights)",
            "config": {"workload": spec.name, "records": bt.B, "memory_rows_per_record": int(bt.lengths.max()),
                       "hidden": shape.H, "questions": schema.Q, "options": schema.O,
                       "l2": "inputs larger than L2 (hidden states %.2f GB per step)" % (hidden.numel() * 2 / 1e9),
                       "parallelism": f"records per GPU, {world} GPU(s)"},
            "memory_tokens_per_s": world * T / (ms / 1e3),
            "roofline": {"bound": "tensor", "kernel": "memory K/V projection GEMM (tcgen05)", "achieved": kv_tf,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": kv_tf / peaks["bf16_tflops"],
                         "peak_source": f"{peak_src} bf16 burst",
                         "frac_of_sustained": kv_tf / peaks["bf16_tflops_sustained"],
                         "traffic": KV_GEMM_TRAFFIC_BYTES, "algorithmic_flops": kv_flops, "ms": kv_ms},
            "kernels": {
                "kv_gemm": {"ms": kv_ms, "tflops": kv_tf, "frac_bf16": kv_tf / peaks["bf16_tflops"]},
                "route_attn_layer1": {"ms": att_ms, "gbs": att_gbs, "frac_hbm": att_gbs / peaks["hbm_gbs"]},
                "span_pool": {"ms": pool_ms, "gbs": pool_gbs, "frac_hbm": pool_gbs / peaks["hbm_gbs"]},
                "row_stats": "computed inside the K/V projection kernel (no pass of its own)",
                "peaks": peaks, "peak_source": peak_src,
            },
            "clocks": clocks.summary(),
            "e2e": {"value": e2e_value, "unit": "records/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "timing": "host wall clock around e2e steps, input copies double-buffered on a copy stream"},
            "gpu_launches": int(launches),
            "stream": stream_info,
            "sharded": sharded,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
