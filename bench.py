"""Benchmark of the PKM lookup forward pass on GB300.

One step = one full forward (scoring, per-half top-k, k^2 merge, softmax,
weighted value read) over one batch of the page-scale workload: B = 16384
queries, H = 4 heads, d_q = 1024, n_keys = 1024 (N = 2^20), d_v = 1024,
k = 32, bf16 inputs, all resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload page|mid|skew|large|tiny|page_fp8|page_layer|
                              page_train|page_train_sparse|mid_flat]

The training workloads add the backward pass to each step; the layer
workload starts from the layer input (query network first); mid_flat
searches all N full keys of the mid workload (the flat exact top-k) and
times the factorised lookup of the same queries beside it.

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload.  This build runs on one GPU: under
torchrun (N > 1) rank 0 prints an "unavailable" line for this arm and no GPU
work is done; the reference arm runs on rank 0 alone.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "PKM lookups (queries×heads)/s; value-gather HBM GB/s and % of GB300 peak"
UNIT = "lookups/s"
L2_FLUSH_BYTES = 512 << 20
# host-buffer calls the pipelined end-to-end measurement keeps in flight: the
# forward workloads use the handle's three staging slots, the layer and
# training workloads two sets of their own device buffers
IN_FLIGHT = 3


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def dist_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload(name, B=None, n_keys=None):
    c = dict(synth.CONFIGS[name])
    if B is not None:
        c["B"] = B
    if n_keys is not None:
        c["n_keys"] = n_keys
    return c


def is_fp8(c):
    return c.get("value_format") == "fp8_e4m3"


def is_train(c):
    """A training workload times the forward and the backward pass."""
    return bool(c.get("train"))


def is_flat(c):
    """A flat workload searches all n_keys^2 full keys instead of the two halves."""
    return bool(c.get("flat"))


def is_layer(c):
    """A layer workload starts from the layer input x and runs the query network."""
    return "qnet_dim" in c


def cpu_inputs(c, sample, C=None, V=None):
    """Inputs of the CPU oracle leg: the first `sample` queries (or layer
    inputs), all tables (an fp8 table quantised by the oracle's own
    quantiser: codes, scales)."""
    import oracle
    if is_layer(c):
        q = synth.query_net_inputs(c, rows=sample)
    else:
        q = synth.queries(c, rows=sample, row_offset=0)
    V = synth.values(c) if V is None else V
    if is_fp8(c):
        V = oracle.quantize_fp8(V, c["n_keys"] ** 2, c["d_v"])
    return q, (synth.subkeys(c) if C is None else C), V


def cpu_oracle_time(c, inputs, sample, nthreads):
    """Wall time of the fp64 oracle forward on `sample` queries of workload c."""
    import oracle
    q, C, V = inputs
    H, d_q, n, d_v, k = c["H"], c["d_q"], c["n_keys"], c["d_v"], c["k"]
    t0 = time.perf_counter()
    if is_layer(c):
        x, W, gamma, beta, mean, var = q
        qf = oracle.query_net(x, W, sample, c["qnet_dim"], H * d_q, gamma, beta, mean, var,
                              c["bn_eps"], nthreads=nthreads)
        q = synth.f32_to_bf16(qf.astype(np.float32))
    if is_fp8(c):
        ref = oracle.lookup(q, C, sample, H, d_q, n, k, nthreads=nthreads)
        oracle.gather_fp8(V[0], V[1], n * n, d_v, ref["idx"], ref["w"], nthreads=nthreads)
    elif is_flat(c):
        # brute force over every full key, then the value read
        idx, score = oracle.brute_topk(q, C, sample, H, d_q, n, k, nthreads=nthreads)
        z = np.exp(score - score[..., :1])
        oracle.gather(V, n * n, d_v, idx, z / z.sum(-1, keepdims=True), nthreads=nthreads)
    elif is_train(c):
        # forward, then the backward pass for its selection (dvalues formed
        # for the selected rows only)
        idx, w, _ = oracle.forward(q, C, V, sample, H, d_q, n, d_v, k, nthreads=nthreads)
        dout = synth.output_grads(c, rows=sample).astype(np.float64)
        oracle.backward(q, C, V, sample, H, d_q, n, d_v, k, idx, w, dout,
                        dvalue_rows=np.unique(idx))
    else:
        oracle.forward(q, C, V, sample, H, d_q, n, d_v, k, nthreads=nthreads)
    return time.perf_counter() - t0


def run_reference(args, rank, world):
    if rank != 0:
        return
    c = workload(args.workload, args.batch, args.n_keys)
    nthreads = os.cpu_count() or 1
    sample = min(args.cpu_sample, c["B"], 64 if is_flat(c) else c["B"])
    inputs = cpu_inputs(c, sample)
    ts = []
    for i in range(args.warmup + args.steps):
        dt = cpu_oracle_time(c, inputs, sample, nthreads)
        if i >= args.warmup:
            ts.append(dt)
    t = sum(ts) / len(ts)
    value = sample * c["H"] / t
    cpu = {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
           "sample": "%d of %d queries of the %s workload per step (fp64 oracle %s)"
                     % (sample, c["B"], args.workload,
                        "forward + backward" if is_train(c)
                        else "brute-force forward" if is_flat(c) else "forward")}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_json(c, args.workload),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def value_row_bytes(c):
    """Bytes of one value row as stored (an fp8 row carries its 4-byte scale)."""
    if is_fp8(c):
        return c["d_v"] + 4
    return c["d_v"] * (2 if c["dtype"] == "bf16" else 4)


def config_json(c, name):
    inputs = "%s, seeded synthetic" % c["dtype"]
    if is_fp8(c):
        inputs = ("bf16 queries and subkeys, seeded synthetic; value table fp8 e4m3 codes with "
                  "per-row fp32 scales, quantised on the GPU from the seeded bf16 table")
    if is_train(c):
        inputs = ("page inputs, seeded synthetic; output gradient dout [B, d_v] fp32 N(0,1); "
                  "step = forward + backward (dq; dsubkeys accumulated in fp32; dvalues %s)"
                  % ("as distinct rows and their fp32 gradient rows" if c.get("sparse_grad")
                     else "accumulated into the dense fp32 table"))
    if is_flat(c):
        inputs = ("mid inputs, seeded synthetic; full key table [H, N, d_q] bf16 materialised "
                  "from the subkeys once, outside the timed steps; step = flat top-k over all "
                  "N full keys + value read")
    if is_layer(c):
        inputs = ("layer input x [B, %d] bf16 N(0,1); query network weight [H*d_q, %d] bf16 "
                  "N(0,1/%d) and BatchNorm running statistics; subkeys and values as page; "
                  "seeded synthetic" % (c["qnet_dim"], c["qnet_dim"], c["qnet_dim"]))
    return {"workload": name, "B": c["B"], "H": c["H"], "d_q": c["d_q"], "n_keys": c["n_keys"],
            "N": c["n_keys"] ** 2, "d_v": c["d_v"], "k": c["k"], "inputs": inputs,
            "l2": "flushed (512 MiB write) between timed steps; value table %.1f GiB"
                  % (c["n_keys"] ** 2 * value_row_bytes(c) / 2**30)}


def run_ours(args, rank, world, local):
    if world > 1:
        # every call of this library runs on one GPU; queries would shard
        # across GPUs as independent replicas, which this build does not run
        # (its tile loads shared by CTA pairs stay on one GPU's memory)
        if rank == 0:
            print(json.dumps({"impl": "ours", "metric": METRIC, "unit": UNIT, "n_gpus": world,
                              "unavailable": "one-GPU build: no multi-GPU path (replicas only, "
                                            "not run)"}), flush=True)
        return
    import torch
    import sparse_top_lookup_gb300 as pk

    torch.cuda.set_device(local)
    c = workload(args.workload, args.batch, args.n_keys)
    if is_flat(c):
        return run_ours_flat(args, c, rank, world)
    B, H, d_q, n, d_v, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "d_v", "k"))
    bf16 = c["dtype"] == "bf16"
    dt = pk.PKM_BF16 if bf16 else pk.PKM_F32
    esz = 2 if bf16 else 4

    # inputs: generated on the host from the seeded streams, copied to HBM once
    def dev(a):
        if bf16:
            return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(a).cuda()

    layer = is_layer(c)
    train = is_train(c)
    C_np, V_np = synth.subkeys(c), synth.values(c)
    dC, dV = dev(C_np), dev(V_np)
    if layer:
        # the layer input and the query network; its BatchNorm is folded once
        dim, F = c["qnet_dim"], H * d_q
        x_np, W_np, *bn = synth.query_net_inputs(c)
        dx, dW = dev(x_np), dev(W_np)
        bn_d = [torch.from_numpy(a).cuda() for a in bn]
        scale, shift = torch.empty(F, device="cuda"), torch.empty(F, device="cuda")
        pk.check(pk.pkm_bn_fold(*bn_d, c["bn_eps"], F, scale, shift), "pkm_bn_fold")
        dq = torch.empty(B, H, d_q, dtype=torch.bfloat16, device="cuda")
    else:
        q_np = synth.queries(c)
        dq = dev(q_np)
    vdt = dt
    if is_fp8(c):
        # the table as stored for the fp8 read: codes then row scales
        dV8 = torch.empty(pk.fp8_table_bytes(n * n, d_v), dtype=torch.uint8, device="cuda")
        pk.check(pk.pkm_quantize_values_fp8(dV, pk.PKM_BF16, n * n, d_v, dV8), "quantize")
        torch.cuda.synchronize()
        dV, vdt = dV8, pk.PKM_FP8_E4M3
    out = torch.empty(B, d_v, device="cuda")
    idx = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
    w = torch.empty(B, H, k, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    cfg = pk.make_config(d_q, d_v, B, H, n, k, q_dtype=dt, value_dtype=vdt, host_staging=1,
                         with_backward=int(train))
    h = pk.pkm_create(cfg)
    if args.select_form is not None:
        pk.check(pk.pkm_set_option(h, pk.PKM_OPT_SELECT_FORM, args.select_form), "set_option")
    stream = torch.cuda.current_stream()
    sparse = bool(c.get("sparse_grad"))
    if train:
        # the backward pass's buffers: dout in, dw between its two calls,
        # gradients out (dsubkeys and a dense dvalues accumulate over the
        # steps; the sparse form rewrites its rows and gradient rows)
        dout_np = synth.output_grads(c)
        g_dout = torch.from_numpy(dout_np).cuda()
        g_dw = torch.empty(B, H, k, device="cuda")
        g_q = torch.empty(B, H, d_q, device="cuda")
        g_C = torch.zeros(H, 2, n, d_q // 2, device="cuda")
        if sparse:
            g_rows = torch.empty(B * H * k, dtype=torch.int64, device="cuda")
            g_grad = torch.empty(B * H * k, d_v, device="cuda")
            g_nrows = torch.zeros(1, dtype=torch.int32, device="cuda")
        else:
            g_V = torch.zeros(n * n, d_v, device="cuda")

    def backward_read():
        if train and sparse:
            pk.check(pk.pkm_backward_read_sparse(h, dV, B, H, n, k, idx, w, g_dout, g_dw, g_rows,
                                                 g_grad, g_nrows, stream),
                     "pkm_backward_read_sparse")
        elif train:
            pk.check(pk.pkm_backward_read(h, dV, B, H, n, k, idx, w, g_dout, g_dw, g_V, stream),
                     "pkm_backward_read")

    def backward_scores():
        if train:
            pk.check(pk.pkm_backward_scores(h, dq, dC, B, H, n, k, idx, w, g_dw, g_q, g_C,
                                            stream), "pkm_backward_scores")

    def qnet():
        if layer:
            pk.check(pk.pkm_query_net(dx, dW, B, dim, F, scale, shift, dq, None, stream),
                     "pkm_query_net")

    def step():
        qnet()
        pk.check(pk.pkm_lookup(h, dq, dC, B, H, n, k, idx, w, stream), "pkm_lookup")
        pk.check(pk.pkm_gather(h, dV, B, H, n, k, idx, w, out, stream), "pkm_gather")
        backward_read()
        backward_scores()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = pk.pkm_get_status(h)
    if st != pk.PKM_OK:
        raise RuntimeError("device status after warm-up: %s" % pk.pkm_strerror(st))

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            qnet()
            ev[i][1].record(stream)
            pk.check(pk.pkm_lookup(h, dq, dC, B, H, n, k, idx, w, stream), "pkm_lookup")
            ev[i][2].record(stream)
            pk.check(pk.pkm_gather(h, dV, B, H, n, k, idx, w, out, stream), "pkm_gather")
            ev[i][3].record(stream)
            backward_read()
            ev[i][4].record(stream)
            backward_scores()
            ev[i][5].record(stream)
        torch.cuda.synchronize()
        # keep sampling clocks long enough to see the load even for short runs
        time.sleep(0.25)
    dist_barrier(world)
    st = pk.pkm_get_status(h)
    if st != pk.PKM_OK:
        raise RuntimeError("device status after timed steps: %s" % pk.pkm_strerror(st))
    # (query, head) pairs of the last timed lookup whose threshold hint missed
    # (their row tiles were selected again without it, inside the step)
    retried = pk.pkm_get_fallback_count(h) if bf16 else 0
    ms_qbatch = None
    if layer:
        # the query network's other BatchNorm mode, timed on the same inputs:
        # the batch's own statistics (two GEMM passes and the statistics)
        qws = torch.empty(pk.pkm_query_net_batch_workspace_bytes(B, F), dtype=torch.uint8,
                          device="cuda")
        q_b = torch.empty_like(dq)

        def qnet_batch():
            pk.check(pk.pkm_query_net_batch(dx, dW, B, dim, F, bn_d[0], bn_d[1], c["bn_eps"],
                                            qws, q_b, None, None, None, stream),
                     "pkm_query_net_batch")
        for _ in range(args.warmup):
            qnet_batch()
        qev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            qev[i][0].record(stream)
            qnet_batch()
            qev[i][1].record(stream)
        torch.cuda.synchronize()
        ms_qbatch = sum(e[0].elapsed_time(e[1]) for e in qev) / args.steps
        del qws, q_b
    t_qnet = [e[0].elapsed_time(e[1]) for e in ev]
    t_lookup = [e[1].elapsed_time(e[2]) for e in ev]
    t_gather = [e[2].elapsed_time(e[3]) for e in ev]
    ms_bread = sum(e[3].elapsed_time(e[4]) for e in ev) / args.steps
    ms_bscores = sum(e[4].elapsed_time(e[5]) for e in ev) / args.steps
    ms_step_local = sum(e[0].elapsed_time(e[5]) for e in ev) / args.steps
    ms_step = dist_max(ms_step_local, world)
    ms_qnet = sum(t_qnet) / args.steps
    ms_lookup = sum(t_lookup) / args.steps
    ms_gather = sum(t_gather) / args.steps

    out_host = torch.empty(B, d_v).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    if train or layer:
        # end to end through the public calls: the step's inputs (q and dout,
        # or the layer input x) in from pinned host memory, the computation
        # (query network; forward; backward), out back to pinned host memory
        # (the gradients stay on the device).  The synchronous form runs one
        # step at a time; the pipelined form keeps two steps in flight, each
        # with its own device copies of the step's tensors, the copies in and
        # out on their own streams
        in_host = torch.from_numpy((x_np if layer else q_np).view(np.int16)).pin_memory()
        dout_host = torch.from_numpy(dout_np).pin_memory() if train else None
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def new_slot():
            sl = {"x": torch.empty_like(dx) if layer else None,
                  "q": torch.empty_like(dq), "out": torch.empty_like(out),
                  "idx": torch.empty_like(idx), "w": torch.empty_like(w),
                  "dout": torch.empty_like(g_dout) if train else None,
                  "oh": torch.empty(B, d_v).pin_memory()}
            for e in ("in", "fwd", "free"):
                sl[e] = torch.cuda.Event()
            return sl
        slots = [new_slot(), new_slot()]

        def step_on(sl, cs):
            # the step's computation on stream cs, from the slot's inputs
            if layer:
                pk.check(pk.pkm_query_net(sl["x"], dW, B, dim, F, scale, shift, sl["q"], None,
                                          cs), "pkm_query_net")
            pk.check(pk.pkm_forward(h, sl["q"], dC, dV, B, H, n, k, sl["out"], sl["idx"],
                                    sl["w"], cs), "pkm_forward")
            sl["fwd"].record(cs)
            if train and sparse:
                pk.check(pk.pkm_backward_sparse(h, sl["q"], dC, dV, B, H, n, k, sl["idx"],
                                                sl["w"], sl["dout"], g_q, g_C, g_rows, g_grad,
                                                g_nrows, cs), "pkm_backward_sparse")
            elif train:
                pk.check(pk.pkm_backward(h, sl["q"], dC, dV, B, H, n, k, sl["idx"], sl["w"],
                                         sl["dout"], g_q, g_C, g_V, cs), "pkm_backward")

        def copy_in(sl):
            dst = sl["x"] if layer else sl["q"]
            dst.view(torch.int16).view(-1).copy_(in_host.view(-1), non_blocking=True)
            if train:
                sl["dout"].copy_(dout_host, non_blocking=True)

        def e2e_call():
            sl = slots[0]
            copy_in(sl)
            step_on(sl, stream)
            sl["oh"].copy_(sl["out"], non_blocking=True)
            stream.synchronize()

        def e2e_pipelined(calls):
            for i in range(calls):
                sl = slots[i % 2]
                if i >= 2:
                    sl["free"].synchronize()  # its host output buffer is reused now
                with torch.cuda.stream(s_in):
                    s_in.wait_event(sl["free"])  # the slot's previous step is done
                    copy_in(sl)
                    sl["in"].record(s_in)
                stream.wait_event(sl["in"])
                step_on(sl, stream)
                comp = torch.cuda.Event()
                comp.record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(sl["fwd"])
                    sl["oh"].copy_(sl["out"], non_blocking=True)
                    s_out.wait_event(comp)
                    sl["free"].record(s_out)
            for sl in slots:
                sl["free"].synchronize()
        h2d = (B * dim * 2) if layer else (B * H * d_q * 2 + B * d_v * 4)
    else:
        # end to end through the host-buffer entry points: every call copies
        # its q in from pinned host memory and its out back; the pipelined
        # form keeps three calls in flight (pkm_forward_host_async, one per
        # staging slot of the handle, three output buffers in turn), the
        # synchronous form one
        q_host = torch.from_numpy(q_np.view(np.int16) if bf16 else q_np).pin_memory()
        out_hosts = [out_host] + [torch.empty(B, d_v).pin_memory() for _ in range(2)]

        def e2e_call():
            pk.check(pk.pkm_forward_host(h, q_host, dC, dV, B, H, n, k, out_host, None, None,
                                         stream), "pkm_forward_host")

        def e2e_pipelined(calls):
            evs = [torch.cuda.Event() for _ in range(calls)]
            for i in range(calls):
                if i >= IN_FLIGHT:
                    evs[i - IN_FLIGHT].synchronize()  # its output buffer is reused now
                pk.check(pk.pkm_forward_host_async(h, q_host, dC, dV, B, H, n, k,
                                                   out_hosts[i % IN_FLIGHT], evs[i],
                                                   stream=stream),
                         "pkm_forward_host_async")
            for ev in evs[-IN_FLIGHT:]:
                ev.synchronize()
        h2d = B * H * d_q * esz
    for _ in range(2):
        e2e_call()
    dist_barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_call()
    e2e_sync_s = dist_max((time.perf_counter() - t0) / e2e_steps, world)
    # several steps (calls) in flight
    e2e_pipelined(4)
    dist_barrier(world)
    t0 = time.perf_counter()
    e2e_pipelined(e2e_steps)
    e2e_s = dist_max((time.perf_counter() - t0) / e2e_steps, world)
    pk.pkm_destroy(h)

    # this host's copy rates on the same pinned buffers (one copy each way,
    # alone), to read the end-to-end figures against
    def copy_gbs(dst, src):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
        b.synchronize()
        return src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
    h_in = in_host if (train or layer) else q_host
    d_tmp = torch.empty_like(h_in, device="cuda")
    copy_gbs(d_tmp, h_in)  # first touches untimed
    copy_gbs(out_host, out)
    h2d_gbs = copy_gbs(d_tmp, h_in)
    d2h_gbs = copy_gbs(out_host, out)
    del d_tmp

    pk_ = peaks()
    gather_bytes = B * H * k * value_row_bytes(c) + B * H * k * 12 + B * d_v * 4
    achieved = gather_bytes / (ms_gather * 1e-3) / 1e9
    flops = 2.0 * B * H * n * d_q
    tflops = flops / (ms_lookup * 1e-3) / 1e12
    value = world * B * H / (ms_step * 1e-3)
    # the value read streams whole rows by bulk copies when the row is a
    # multiple of 512 bytes (every bench workload), else one CTA per query
    code_row = d_v * (1 if is_fp8(c) else esz)
    gather_name = ("gather_bulk_kernel" if code_row % 512 == 0 and code_row <= 8192
                   else "gather_kernel")
    traffic = measured_traffic(args.workload, B, gather_name)
    roof = {"kernel": "%s (value read)" % gather_name, "bound": "hbm",
            "achieved": achieved, "peak": pk_["hbm"], "unit": "GB/s",
            "frac": achieved / pk_["hbm"], "traffic": traffic, "peak_source": pk_["src"],
            # distinct value rows the step selected (each crosses HBM at most
            # once per launch if L2 keeps it), and the DRAM rate of the
            # measured traffic when a profile of this source and batch exists
            "distinct_rows": int(torch.unique(idx).numel()),
            "dram_gbs": traffic / (ms_gather * 1e-3) / 1e9 if traffic else None}
    if train:
        # per distinct selected row: the value row read once and its dvalues
        # row read and written once (fp32; the sparse form writes its gradient
        # row and row number once); per selection: idx, w and dw; per query:
        # dout.  The time is the whole read call (bucket count, scan and
        # scatter, sort, then row_grad_kernel).
        rows_touched = roof["distinct_rows"]
        per_row = value_row_bytes(c) + (4 * d_v + 8 if sparse else 8 * d_v)
        bread_bytes = rows_touched * per_row + B * H * k * 16 + B * d_v * 4
        bread = bread_bytes / (ms_bread * 1e-3) / 1e9
        broof = {"kernel": "pkm_backward_read%s (bucket sort + row_grad_kernel)"
                 % ("_sparse" if sparse else ""), "bound": "hbm",
                 "achieved": bread, "peak": pk_["hbm"], "unit": "GB/s",
                 "frac": bread / pk_["hbm"],
                 "traffic": measured_traffic(args.workload, B, "row_grad_kernel", "backward.cu"),
                 "peak_source": pk_["src"],
                 "rows_touched": rows_touched}
        forward_roof, roof = roof, broof
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": c["dtype"], "data": "synthetic",
        "config": config_json(c, args.workload),
        "queries_per_s": world * B / (ms_step * 1e-3),
        "stages_ms": (({"query_net": ms_qnet} if layer else {}) |
                      {"lookup": ms_lookup, "gather": ms_gather} |
                      ({"backward_read": ms_bread, "backward_scores": ms_bscores}
                       if train else {})),
        "roofline": roof,
        "retried_pairs": retried,
        "scoring_roofline": {"kernel": "select_2sm_kernel + merge_kernel (a1-a5, one lookup call)",
                             "bound": "tensor", "achieved": tflops, "peak": pk_["bf16"],
                             "unit": "TFLOP/s", "frac": tflops / pk_["bf16"],
                             "peak_source": pk_["src"] + " bf16 burst"},
        "e2e": {"value": world * B * H / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": B * d_v * 4,
                "calls_in_flight": 2 if (train or layer) else IN_FLIGHT,
                "copy_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs},
                "value_one_call_in_flight": world * B * H / e2e_sync_s},
        # per step: select_2sm_kernel and merge_kernel, their retry launches
        # (return at once when no row missed its threshold hint) and the
        # value read (fp32 inputs: lookup_simt_kernel and the value read)
        # (training: bucket_count, bucket_scan, bucket_scatter, bucket_sort
        # and row_grad kernels, zero_rows for the sparse gradient, and
        # ds_gather, key_scan, key_scatter and dsub kernels too, besides
        # memsets)
        "gpu_launches": ((5 if bf16 else 2) + (1 if layer else 0)
                         + ((10 if sparse else 9) if train else 0)) * args.steps,
        "clocks": clk.summary(),
    }
    if train:
        line["forward_roofline"] = forward_roof
    if layer:
        qflops = 2.0 * B * dim * F
        line["query_net_roofline"] = {
            "kernel": "qnet_kernel (x W^T + BatchNorm, tcgen05)", "bound": "tensor",
            "achieved": qflops / (ms_qnet * 1e-3) / 1e12, "peak": pk_["bf16"], "unit": "TFLOP/s",
            "frac": qflops / (ms_qnet * 1e-3) / 1e12 / pk_["bf16"],
            "peak_source": pk_["src"] + " bf16 burst"}
        line["query_net_modes_ms"] = {
            "running_stats": ms_qnet, "batch_stats": ms_qbatch,
            "batch_stats_note": "statistics pass (GEMM with column-statistics epilogue), the "
                                "blocks joined by the law of total variance, then the GEMM "
                                "again with the folded scale and shift; timed after the steps, "
                                "not part of them"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        sample = min(args.cpu_sample, B)
        inputs = cpu_inputs(c, sample, C=C_np, V=V_np)
        t = cpu_oracle_time(c, inputs, sample, nthreads)
        # the same oracle on one thread, on the first quarter of the sample
        s1 = max(1, sample // 4)
        q_in = inputs[0]
        if is_layer(c):
            q1 = (q_in[0][: s1 * c["qnet_dim"]],) + tuple(q_in[1:])
        else:
            q1 = q_in[: s1 * H * d_q]
        t1 = cpu_oracle_time(c, (q1,) + tuple(inputs[1:]), s1, 1)
        line["cpu_baseline"] = {
            "value": sample * H / t, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": "%d of %d queries (all %d heads) of the %s workload, fp64 oracle %s"
                      % (sample, B, H, args.workload,
                         "forward + backward" if train else "forward"),
            "value_1_thread": s1 * H / t1, "sample_1_thread": "the first %d of them" % s1}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ours_flat(args, c, rank, world):
    """The flat forward: per step the exact top-k over all N = n_keys^2 full
    keys (pkm_flat_lookup) and the value read; the factorised lookup of the
    same queries is timed in the same run for the comparison."""
    import torch
    import sparse_top_lookup_gb300 as pk

    B, H, d_q, n, d_v, k = (c[x] for x in ("B", "H", "d_q", "n_keys", "d_v", "k"))
    N = n * n

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)

    q_np, C_np, V_np = synth.queries(c), synth.subkeys(c), synth.values(c)
    dq, dC, dV = dev(q_np), dev(C_np), dev(V_np)
    out = torch.empty(B, d_v, device="cuda")
    idx = torch.empty(B, H, k, dtype=torch.int64, device="cuda")
    w = torch.empty(B, H, k, device="cuda")
    fidx, fw = torch.empty_like(idx), torch.empty_like(w)
    keys = torch.empty(H, N, d_q, dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    h = pk.pkm_create(pk.make_config(d_q, d_v, B, H, n, k))
    stream = torch.cuda.current_stream()
    # the full key table, once (as a value table is written once)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pk.check(pk.pkm_full_keys(h, dC, H, n, keys, stream), "pkm_full_keys")
    e1.record(stream)
    torch.cuda.synchronize()
    ms_keys = e0.elapsed_time(e1)

    def flat_step():
        pk.check(pk.pkm_flat_lookup(h, dq, keys, B, H, n, k, idx, w, stream), "pkm_flat_lookup")
        pk.check(pk.pkm_gather(h, dV, B, H, n, k, idx, w, out, stream), "pkm_gather")

    for _ in range(args.warmup):
        flush.zero_()
        flat_step()
        pk.check(pk.pkm_lookup(h, dq, dC, B, H, n, k, fidx, fw, stream), "pkm_lookup")
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            pk.check(pk.pkm_flat_lookup(h, dq, keys, B, H, n, k, idx, w, stream),
                     "pkm_flat_lookup")
            ev[i][1].record(stream)
            pk.check(pk.pkm_gather(h, dV, B, H, n, k, idx, w, out, stream), "pkm_gather")
            ev[i][2].record(stream)
        # the factorised search of the same queries, for the comparison
        for i in range(args.steps):
            flush.zero_()
            fev[i][0].record(stream)
            pk.check(pk.pkm_lookup(h, dq, dC, B, H, n, k, fidx, fw, stream), "pkm_lookup")
            fev[i][1].record(stream)
        torch.cuda.synchronize()
        time.sleep(0.25)
    dist_barrier(world)
    st = pk.pkm_get_status(h)
    if st != pk.PKM_OK:
        raise RuntimeError("device status after timed steps: %s" % pk.pkm_strerror(st))
    ms_flat = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    ms_gather = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    ms_step = dist_max(sum(e[0].elapsed_time(e[2]) for e in ev) / args.steps, world)
    ms_fact = sum(e[0].elapsed_time(e[1]) for e in fev) / args.steps
    same = float((idx == fidx).all(-1).float().mean())

    # end to end: q in from pinned host memory, flat lookup and read, out back
    q_host = torch.from_numpy(q_np.view(np.int16)).pin_memory()
    out_host = torch.empty(B, d_v).pin_memory()

    def e2e_call():
        dq.view(torch.int16).view(-1).copy_(q_host.view(-1), non_blocking=True)
        flat_step()
        out_host.copy_(out, non_blocking=True)
        stream.synchronize()
    for _ in range(2):
        e2e_call()
    e2e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_call()
    e2e_s = dist_max((time.perf_counter() - t0) / e2e_steps, world)
    pk.pkm_destroy(h)

    pk_ = peaks()
    flops = 2.0 * B * H * N * d_q
    tflops = flops / (ms_flat * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": world * B * H / (ms_step * 1e-3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": c["dtype"],
        "data": "synthetic", "config": config_json(c, args.workload),
        "queries_per_s": world * B / (ms_step * 1e-3),
        "stages_ms": {"flat_lookup": ms_flat, "gather": ms_gather},
        "roofline": {"kernel": "select_2sm_kernel, flat form (scoring of all N full keys and "
                               "the exact top-k)", "bound": "tensor", "achieved": tflops,
                     "peak": pk_["bf16"], "unit": "TFLOP/s", "frac": tflops / pk_["bf16"],
                     "traffic": None, "peak_source": pk_["src"] + " bf16 burst"},
        "flat_vs_factorised": {
            "flat_lookup_ms": ms_flat, "factorised_lookup_ms": ms_fact,
            "time_ratio": ms_flat / ms_fact,
            "key_comparisons_per_query_head": {"flat": N, "factorised": 2 * n},
            "comparison_ratio": N / (2 * n),
            "page_counts": "the pages' worked example: 2048 subkey comparisons instead of "
                           "10^6 at N = 10^6, k = 32",
            "same_selection_frac": same,
            "full_keys_ms": ms_keys, "full_keys_bytes": H * N * d_q * 2},
        "e2e": {"value": world * B * H / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": B * H * d_q * 2, "d2h_bytes_per_step": B * d_v * 4,
                "calls_in_flight": 1},
        # per step: select_2sm_kernel (flat form) and the value read
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        sample = min(args.cpu_sample, 64, B)
        inputs = cpu_inputs(c, sample, C=C_np, V=V_np)
        t = cpu_oracle_time(c, inputs, sample, nthreads)
        line["cpu_baseline"] = {
            "value": sample * H / t, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": "%d of %d queries (all %d heads) of the %s workload, fp64 oracle brute "
                      "force over all N full keys + value read" % (sample, B, H, args.workload)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def measured_traffic(workload_name, B, kernel="gather_bulk_kernel", source="gather.cu"):
    """DRAM bytes (read + write) of one launch (or call) from the committed ncu
    summary profiles/<kernel>_<workload>.md, if it was taken on this workload
    and the kernel source is unchanged since (its sha256 prefix is recorded);
    else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel, workload_name))
    src = os.path.join(ROOT, "sparse_top_lookup_gb300", "csrc", source)
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if line.startswith("- ") and ": " in line:
            key, val = line[2:].split(": ", 1)
            fields[key.strip()] = val.strip().strip("`")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if fields.get("source sha256") != sha or fields.get("B") != str(B):
        return None
    try:
        return int(fields["dram bytes read"]) + int(fields["dram bytes written"])
    except (KeyError, ValueError):
        return None



def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="page", choices=sorted(synth.CONFIGS))
    ap.add_argument("--cpu-sample", type=int, default=1024)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's query count B (profiling runs)")
    ap.add_argument("--n-keys", type=int, default=None,
                    help="override the workload's n_keys (small profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--select-form", type=int, default=None, choices=[0, 1, 2, 3],
                    help="selection kernel form of the bf16 lookup (PKM_OPT_SELECT_FORM)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
