#!/usr/bin/env python3
"""Benchmark of the rotated INT2 KV-cache decode step on GB300.

Workload (default, the 32K-context configuration): 8B-class GQA layer, 32 query
heads / 8 KV heads, head dim 128, hidden 4096, bf16 inputs, 16 sequences x
32,768 tokens in a paged INT2 cache (16-token pages, shuffled block table),
per-head dense learned-style rotations R = expm(A - A^T), key mean subtracted.

One step = the whole hot path for one decode token of every sequence:
  1. kvq_decode_step -- the query preparation rotates, centres, clips, quantizes,
                        packs and writes the new token's K and V (position 32,767)
                        and rotates the query; split-K attention over 32,768 packed
                        tokens; log-sum-exp combine
  2. kvq_out_proj_packed -- y = o' W_O-bar^T with R_V folded into W_O (W_O-bar stored in
                        the projection's box order by kvq_pack_wo)
(with --window, kvq_decode_step_win also writes the new token's BF16 window copy
and the decode reads the windows)
value = sequences x steps / time (decode tokens per second, one layer).

--impl reference times the fp64 oracle (CPU) on a bounded sample of the same
workload.  --case append_chunk / calib time the 4,096-token prefill append and
the calibration sweep instead (for profiling; not the headline line).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT2 decode attention: KV-cache GB/s read (% of HBM peak), tokens/s at 32K ctx"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
MIN_TIMED_S = 0.5  # the timed region repeats its block of steps until it spans this long
MAX_BLOCKS = 100000


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    p.add_argument("--case", choices=["decode_step", "append_chunk", "append_chunk_dense", "calib", "report", "optr"],
                   default="decode_step")
    p.add_argument("--workload", choices=["gqa8b", "long4b", "serve14b"], default="gqa8b",
                   help="decode-step shape: gqa8b (default, the headline), long4b (128K), serve14b (ragged)")
    p.add_argument("--seqs", type=int, default=None, help="sequences (default: 16 gqa8b, 1 long4b, 64 serve14b)")
    p.add_argument("--ctx", type=int, default=None, help="context (gqa8b default 32768, long4b 131072)")
    p.add_argument("--splits", type=int, default=0)
    p.add_argument("--page", type=int, choices=[8, 16], default=None, help="tokens per page (default 16)")
    p.add_argument("--clips", default=None, metavar="K,V",
                   help="clip ratios of keys and values, e.g. 0.96,0.92 (Table A); default per workload")
    p.add_argument("--window", default=None, metavar="SINK,RECENT",
                   help="decode step with BF16 sink / recent windows, e.g. 64,256 (default: all tokens INT2)")
    p.add_argument("--optr-steps", type=int, default=80, help="--case optr: Adam steps per phase (the paper: 80)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons; only the samples
    whose timestamps fall inside the timed region are reported."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True, interval_ms: int = 20):
        self.proc = None
        self.t0 = self.t1 = None
        if enabled:
            sel = str(device_index)
            try:
                import torch
                uuid = str(getattr(torch.cuda.get_device_properties(device_index), "uuid", "") or "")
                if uuid:
                    sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            except Exception:
                pass
            try:
                self.proc = subprocess.Popen(["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}",
                                              "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.5)  # let the sampler start before the timed region
            except Exception:
                self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        import datetime
        sm, mx, reasons, n_all = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(f[1]), float(f[2])
            except ValueError:
                continue
            n_all += 1
            if self.t0 is None or not (self.t0 <= ts <= self.t1):
                continue
            sm.append(clk)
            mx = cmax
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window_s": round(self.t1 - self.t0, 3)}


def traffic_record(kernel_file: str, key: str):
    """Per-launch DRAM traffic from a committed ncu summary, valid only for the
    workload named in the key and while the kernel source is unchanged (the
    summary stores the source's sha256); None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "int2_kv_cache_gb300", "csrc", kernel_file)
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for line in open(path):
            f = line.split()
            if len(f) >= 3 and f[0] == key and f[2] == digest:
                return float(f[1])
    except OSError:
        pass
    return None


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gen_parallel(fn, n):
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        return list(ex.map(fn, range(n)))


def decode_workload(args):
    """The decode case named by --workload (sizes from --seqs / --ctx when given)."""
    from int2_kv_cache_gb300 import workloads as W
    kw = {}
    if args.page:
        kw["page_tokens"] = args.page
    if args.clips:
        kw["clip_k"], kw["clip_v"] = (float(x) for x in args.clips.split(","))
    if args.workload == "long4b":
        return W.long4b_128k(n_seqs=args.seqs or 1, ctx=args.ctx or 131072, **kw)
    if args.workload == "serve14b":
        return W.serve14b_ragged(n_seqs=args.seqs or 64, **kw)
    return W.gqa8b_32k(n_seqs=args.seqs or 16, ctx=args.ctx or 32768, **kw)


def workload_text(c) -> str:
    lens = np.asarray(c.seq_lens)
    ctx = f"ctx {int(lens[0])}" if lens.min() == lens.max() else f"ragged ctx {int(lens.min())}..{int(lens.max())}"
    rot = {"dense": "dense expm(A-A^T)", "signed_hadamard": "signed-Hadamard", "identity": "identity"}[c.rot_k.kind]
    clip = (f"clip {float(c.clip_k):g}" if c.clip_k == c.clip_v else
            f"clips K {float(c.clip_k):g} / V {float(c.clip_v):g}")
    return (f"{c.name.split('_')[0]} decode step: B={len(lens)} x {ctx}, Hq {c.n_q_heads} / Hkv {c.n_kv_heads}, "
            f"d 128, hidden {c.d_model}, {c.page_tokens}-token pages (shuffled), {rot} rotations, mu-centred keys, "
            f"{clip}")


class DecodeStep:
    """The decode-step workload resident on one GPU: every sequence holds len - 1
    cached tokens; a step appends its last token, decodes over len tokens and
    projects through the folded W_O."""

    def __init__(self, c, splits: int, device: str, window=None):
        import torch
        import int2_kv_cache_gb300 as kvq

        self.torch, self.kvq, self.dev = torch, kvq, device
        self.case = c
        lens = np.asarray(c.seq_lens, dtype=np.int64)
        n_seqs = len(lens)
        self.lens_np = lens
        self.B, self.L, self.hq, self.hkv, self.dm = n_seqs, int(lens.max()), c.n_q_heads, c.n_kv_heads, c.d_model
        ctx = self.L
        bf = torch.bfloat16
        t = lambda x, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(x)).to(device).to(dt)
        self.t = t
        self.layout = kvq.make_layout(c.page_tokens, c.n_kv_heads, c.n_q_heads, c.num_blocks, c.block_table.shape[1])
        self.table = t(c.block_table, torch.int32)
        self.rot_k = kvq.DeviceRot.from_spec(c.rot_k, device)
        self.rot_v = kvq.DeviceRot.from_spec(c.rot_v, device)
        # key mean (Eq. 19) and its rotation (Eq. 20), on the GPU
        mu = torch.empty(c.n_kv_heads, 128, device=device)
        kvq.kvq_key_mean(t(c.calibration_keys(), bf), mu)
        self.mu_rot = torch.empty_like(mu)
        kvq.kvq_rotate_heads(mu.reshape(1, c.n_kv_heads, 128), self.rot_k, self.mu_rot.reshape(1, c.n_kv_heads, 128))
        # paged cache: positions 0 .. len-2 are history; every step writes position len-1
        self.pool = torch.zeros(kvq.kvq_pool_bytes(self.layout), dtype=torch.uint8, device=device)
        for b0 in range(0, n_seqs, 4):
            kvs = gen_parallel(lambda i: c.kv(b0 + i), min(4, n_seqs - b0))
            for i, (k, v) in enumerate(kvs):
                b = b0 + i
                hist = int(lens[b]) - 1
                kvq.kvq_quantize_append(self.layout, t(k[:hist], bf), t(v[:hist], bf), t(np.array([0, hist]), torch.int32),
                                        t(np.array([0]), torch.int32), self.table[b:b + 1].contiguous(), self.rot_k,
                                        self.rot_v, self.mu_rot, c.clip_k, c.clip_v, self.pool)
        # BF16 sink / recent windows: the window copies of the history
        self.win = None
        self.mu = mu
        if window is not None:
            s_w, r_w = window
            self.win = kvq.Window(s_w, r_w, torch.zeros(kvq.Window.buffer_bytes(n_seqs, c.n_kv_heads, s_w, r_w),
                                                        dtype=torch.uint8, device=device))
            for b0 in range(0, n_seqs, 4):
                kvs = gen_parallel(lambda i: c.kv(b0 + i), min(4, n_seqs - b0))
                for i, (k, v) in enumerate(kvs):
                    b = b0 + i
                    hist = int(lens[b]) - 1
                    # only the tokens that end up in a window are needed: the sink and the last r_w
                    for lo, hi in ((0, min(s_w, hist)), (max(s_w, hist - r_w), hist)):
                        if hi <= lo:
                            continue
                        kvq.kvq_window_append(self.layout, t(k[lo:hi], bf), t(v[lo:hi], bf),
                                              t(np.array([0, hi - lo]), torch.int32), t(np.array([lo]), torch.int32),
                                              mu, self.win_row(b))
        torch.cuda.synchronize()
        kvq.kvq_device_check()
        # folded W_O (Eqs. 29-31), bf16
        self.w_fold = torch.empty(self.dm, self.hq * 128, dtype=bf, device=device)
        kvq.kvq_fold_wo(t(c.w_o(), bf), self.hq, self.hkv, self.rot_v, self.w_fold)
        # the projection's box order (one contiguous 16 KB DRAM stream per tensor-core box)
        self.w_pack = torch.empty(kvq.kvq_wo_packed_bytes(self.dm, self.hq * 128), dtype=torch.uint8, device=device)
        kvq.kvq_pack_wo(self.w_fold, self.w_pack)
        # step inputs
        kn, vn = zip(*[c.new_kv(b, 1) for b in range(n_seqs)])
        # the step's inputs (q, new K, new V) staged in one pinned buffer: one host->device copy per step
        parts = [c.queries(), np.concatenate(kn), np.concatenate(vn)]
        sizes = [x.size for x in parts]
        self.host_in = torch.empty(sum(sizes), dtype=bf).pin_memory()
        o = 0
        for x in parts:
            self.host_in[o:o + x.size] = torch.from_numpy(np.ascontiguousarray(x).reshape(-1)).to(bf)
            o += x.size
        self.dev_in = self.host_in.to(device)
        views, o = [], 0
        for x in parts:
            views.append(self.dev_in[o:o + x.size].view(x.shape))
            o += x.size
        self.q, self.k_new, self.v_new = views
        # the same inputs as views of the pinned host buffer: the end-to-end steps hand these
        # host pointers to the API (the query preparation reads them over the host link)
        hv, o = [], 0
        for x in parts:
            hv.append(self.host_in[o:o + x.size].view(x.shape))
            o += x.size
        self.host_q, self.host_k_new, self.host_v_new = hv
        self.cu_new = t(np.arange(n_seqs + 1), torch.int32)
        self.start = t(lens - 1, torch.int32)
        self.lens = t(lens, torch.int32)
        self.splits = splits
        ws = kvq.kvq_decode_workspace_size_win(self.layout, n_seqs, ctx, self.win, splits)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        # work partitions of 4 warps of the decode kernel (the library's choice when splits == 0)
        self.n_ctas = splits or next(s for s in range(1, 8193)
                                     if kvq.kvq_decode_workspace_size_win(self.layout, n_seqs, ctx, self.win, s) == ws)
        self.o = torch.empty(n_seqs, self.hq, 128, device=device)
        self.y = torch.empty(n_seqs, self.dm, device=device)
        self.host_y = torch.empty(n_seqs, self.dm).pin_memory()
        # the fused step (query prep with the append (and window copy), decode, combine) + W_O
        self.launches_per_step = 3 + 1

    def win_row(self, b):
        """A window struct over sequence b's rows only (for appending one sequence at a time)."""
        w = self.win
        per = self.kvq.Window.buffer_bytes(1, self.case.n_kv_heads, w.sink_tokens, w.recent_tokens)
        return self.kvq.Window(w.sink_tokens, w.recent_tokens, w.buf[b * per:(b + 1) * per])

    def step(self, ev=None, host_io=False):
        """One decode step: kvq_decode_step (the new token's append fused into the decode
        call; with windows kvq_decode_step_win, which also writes its window copy) and the
        W_O projection.  ev: events [4] recorded before the step, before the decode call
        (the same point), after it and after the projection.  host_io: read q and the new
        K/V from the pinned host buffer and write y into pinned host memory (the kernels
        move the bytes over the host link themselves)."""
        kvq = self.kvq
        c = self.case
        q, k_new, v_new, y = ((self.host_q, self.host_k_new, self.host_v_new, self.host_y) if host_io
                              else (self.q, self.k_new, self.v_new, self.y))
        if ev is not None:
            ev[0].record()
            ev[1].record()
        if self.win is None:
            kvq.kvq_decode_step(self.layout, q, k_new, v_new, self.lens, self.L, self.table, self.rot_k,
                                self.rot_v, self.mu_rot, c.clip_k, c.clip_v, self.pool, self.ws, self.o,
                                n_splits=self.splits)
        else:
            kvq.kvq_decode_step_win(self.layout, q, k_new, v_new, self.lens, self.L, self.table,
                                    self.rot_k, self.rot_v, self.mu_rot, self.mu, c.clip_k, c.clip_v, self.pool,
                                    self.win, self.ws, self.o, n_splits=self.splits)
        if ev is not None:
            ev[2].record()
        kvq.kvq_out_proj_packed(self.o.reshape(self.B, -1), self.w_pack, y, self.dm)
        if ev is not None:
            ev[3].record()

    def decode_only(self, ev):
        """kvq_decode_attention alone over the same cache (for the per-phase record)."""
        ev[0].record()
        self.kvq.kvq_decode_attention(self.layout, self.q, self.lens, self.L, self.table, self.rot_k, self.pool,
                                      self.ws, self.o, n_splits=self.splits)
        ev[1].record()

    def step_e2e(self):
        """A step whose inputs are in pinned host memory and whose output goes there: the
        API gets the host pointers, so the query preparation reads q and the new K/V, and
        the projection writes y, across the host link inside the step (no staging copies)."""
        self.step(host_io=True)

    def decode_bytes(self) -> dict:
        B, hq, hkv = self.B, self.hq, self.hkv
        lens = self.lens_np
        g = hq // hkv
        units = B * hkv
        frag = ((g + 3) // 4) * 16 * 32 * 4
        if self.win is not None:
            # INT2 positions [S, L - R) read at 72 bytes, window positions at 512 (bf16 key + value)
            s_w, r_w = self.win.sink_tokens, self.win.recent_tokens
            n_win = np.minimum(lens, s_w) + np.maximum(0, lens - np.maximum(s_w, lens - r_w))
            n_int2 = lens - n_win
            pairs = min(4 * self.n_ctas + units, int(hkv * ((n_int2 + 63) // 64).sum()))
            pairs_w = min(4 * self.n_ctas + units, int(hkv * ((n_win + 7) // 8 + 1).sum()))
            return {
                "kv_cache": int(n_int2.sum()) * hkv * 72,
                "bf16_windows": int(n_win.sum()) * hkv * 512,
                "q": B * hq * 128 * 2,
                "block_table": int(((n_int2 + self.case.page_tokens - 1) // self.case.page_tokens).sum()) * 4,
                "rotation": hkv * 128 * 128 * 4,
                "query_fragments_write_read": 2 * units * (2 * frag + g * 16),
                "partials_write_read": 2 * (pairs + pairs_w) * g * 130 * 4,
                "o_rot": B * hq * 128 * 4,
                # the step's new token: bf16 K and V read, 72 B of codes and meta and 512 B of
                # window row written per head, R_V read
                "step_append": B * hkv * (2 * 256 + 72 + 512) + (hkv * 128 * 128 * 4
                                                               if self.case.rot_v.kind == "dense" else hkv * 128 * 4),
            }
        # one partial (acc[128], m, l per query head) per (warp slice, unit) pair:
        # at most 4 * n_ctas + units of them, written once and read once
        pairs = min(4 * self.n_ctas + units, int(hkv * ((lens + 63) // 64).sum()))
        cache = int(lens.sum()) * hkv * 72
        dense_v = self.case.rot_v.kind == "dense"
        return {
            "kv_cache": cache,
            # the step's new token: bf16 K and V read, 72 B of codes and meta written, R_V read
            "step_append": B * hkv * (2 * 256 + 72) + (hkv * 128 * 128 * 4 if dense_v else hkv * 128 * 4),
            "q": B * hq * 128 * 2,
            "block_table": int(((lens + self.case.page_tokens - 1) // self.case.page_tokens).sum()) * 4,
            "rotation": hkv * 128 * 128 * 4,
            "query_fragments_write_read": 2 * units * (((g + 3) // 4) * 16 * 32 * 4 + g * 16),
            "partials_write_read": 2 * pairs * g * 130 * 4,
            "o_rot": B * hq * 128 * 4,
        }


def run_gpu(args):
    import torch
    from int2_kv_cache_gb300 import _build
    _build.build()
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    window = tuple(int(x) for x in args.window.split(",")) if args.window else None
    w = DecodeStep(decode_workload(args), args.splits, device, window)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        w.step()
    barrier()
    # the timed steps: no events between the phases (they would split the
    # programmatic dependent launches that chain the decode and projection kernels).
    # Blocks of exactly `steps` steps, each bracketed by events, are repeated until
    # the timed region spans at least MIN_TIMED_S (so the clock sampler sees it);
    # the step time is the median over the blocks.
    clocks = Clocks(local, enabled=not args.no_clocks)
    barrier()
    clocks.mark_start()
    t_wall = time.perf_counter()
    block_ms = []
    while True:
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(args.steps):
            w.step()
        stop.record(stream)
        stop.synchronize()
        block_ms.append(start.elapsed_time(stop))
        if time.perf_counter() - t_wall >= MIN_TIMED_S or len(block_ms) >= MAX_BLOCKS:
            break
    barrier()
    clocks.mark_stop()
    clk = clocks.stop()
    total_ms = float(np.median(block_ms))
    # per-phase breakdown (separate steps, events around each entry point)
    n_br = max(min(args.steps * len(block_ms), 400), 20)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_br)]
    for i in range(n_br):
        w.step(evs[i])
    barrier()
    t_dec = float(np.median([e[1].elapsed_time(e[2]) for e in evs]))
    t_out = float(np.median([e[2].elapsed_time(e[3]) for e in evs]))
    t_dec_only = None
    if window is None:
        # kvq_decode_attention alone over the same cache (no append), for the record
        evd = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_br)]
        for i in range(n_br):
            w.decode_only(evd[i])
        barrier()
        t_dec_only = float(np.median([e[0].elapsed_time(e[1]) for e in evd]))

    # end to end through the public API with host buffers
    for _ in range(3):
        w.step_e2e()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        w.step_e2e()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    w.kvq.kvq_device_check()

    ms = torch.tensor([total_ms / args.steps, e2e_ms], device=device)
    if world > 1:
        torch.distributed.all_reduce(ms, op=torch.distributed.ReduceOp.MAX)
    ms_step, e2e_step = float(ms[0]), float(ms[1])
    if rank != 0:
        return
    peak, peak_kind = peaks()
    by = w.decode_bytes()
    alg = sum(by.values())
    achieved = alg / (t_dec * 1e-3) / 1e9
    traffic = traffic_record("decode.cu", "decode_step_" + args.workload) if window is None else None
    line = {
        "metric": METRIC,
        "value": world * w.B / (ms_step * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "timed_blocks": len(block_ms),
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; bf16 q/K/V/W_O, 2-bit cache)",
        "config": {
            "workload": workload_text(w.case),
            "batch": w.B, "ctx": w.L, "n_q_heads": w.hq, "n_kv_heads": w.hkv, "d_model": w.dm,
            "decode_warps": 4 * w.n_ctas, "parallelism": f"replicas x{world}",
            "bf16_windows": (f"sink {window[0]} + recent {window[1]} tokens per sequence in BF16"
                             if window else "none (every token INT2)"),
            "l2": "inputs larger than L2 (KV pool %.0f MB > 129 MB); no flush" % (w.pool.numel() / 1e6),
        },
        "kernel_ms": ({"decode_step": t_dec, "out_proj": t_out, "decode_attention_alone": t_dec_only}
                      if window is None else
                      {"decode_step_win": t_dec, "out_proj": t_out}),
        "kv_cache_gbs": by["kv_cache"] / (t_dec * 1e-3) / 1e9,
        "kv_cache_pct_of_peak": {"measured": by["kv_cache"] / (t_dec * 1e-3) / 1e9 / peak,
                                 "nominal_8tbs": by["kv_cache"] / (t_dec * 1e-3) / 1e9 / NOMINAL_HBM_GBS},
        "roofline": {"kernel": ("kvq_decode_step (query prep with the new token's append, decode, combine)"
                                if window is None else
                                "kvq_decode_step_win (query prep with the new token's append and window copy, "
                                "decode, combine)"),
                     "bound": "hbm", "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes": alg, "bytes": by},
        "e2e": {"value": world * w.B / (e2e_step * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(w.host_in.numel() * 2),
                "d2h_bytes_per_step": int(w.host_y.numel() * 4),
                "transfer": "q and the new K/V read from pinned host memory by the query preparation, y written "
                            "to pinned host memory by the projection (host pointers through the C ABI)"},
        "gpu_launches": w.launches_per_step * args.steps * len(block_ms),
        "clocks": clk,
    }
    # the prefill-chunk quantize-append (4 x 4,096 tokens, 4B-class layer), its own roofline
    line["append_chunk"] = append_chunk_measure(device, False, 50, 5, min_s=0.25)
    # the same chunk with dense learned rotations (8B-class layer): the tensor-core cache write
    line["append_chunk_dense"] = append_chunk_measure(device, True, 20, 3, min_s=0.25)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w.case, budget_s=12.0)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and --impl reference)
# ---------------------------------------------------------------------------

class OracleStep:
    """The fp64 oracle doing one decode step for one sequence of the workload."""

    def __init__(self, case, b: int = 0):
        import oracle
        self.o = oracle
        c = case
        self.c, self.b = c, b
        self.r_k = oracle.rotations.rot_matrices(c.rot_k, c.n_kv_heads)
        self.r_v = oracle.rotations.rot_matrices(c.rot_v, c.n_kv_heads)
        self.mu = oracle.cache.key_mean(c.calibration_keys())
        self.w_fold = oracle.output.fold_wo(c.w_o(), self.r_v, c.gqa)
        k, v = c.kv(b)
        self.L = int(c.seq_lens[b])
        hist = self.L - 1
        self.pool = np.zeros(oracle.cache.pool_bytes(c.num_blocks, c.n_kv_heads, c.page_tokens), np.uint8)
        enc = oracle.cache.encode_tokens(k[:hist], v[:hist], self.r_k, self.r_v, self.mu, c.clip_k, c.clip_v)
        oracle.cache.write_tokens(self.pool, c.n_kv_heads, c.page_tokens, c.block_table[b], 0, enc)
        self.k_new, self.v_new = c.new_kv(b, 1)
        self.q = c.queries()[b]

    def step(self):
        o, c = self.o, self.c
        enc = o.cache.encode_tokens(self.k_new, self.v_new, self.r_k, self.r_v, self.mu, c.clip_k, c.clip_v)
        o.cache.write_tokens(self.pool, c.n_kv_heads, c.page_tokens, c.block_table[self.b], self.L - 1, enc)
        kh, vh = o.cache.dequantized_sequence(self.pool, c.n_kv_heads, c.page_tokens, c.block_table[self.b], self.L)
        o_rot = o.attention.decode_attention(self.q, kh, vh, self.r_k, c.gqa)
        return o.output.out_proj(o_rot, self.w_fold)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(case, budget_s: float = 12.0) -> dict:
    st = OracleStep(case, 0)
    n, t0 = 0, time.perf_counter()
    while True:
        st.step()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 50:
            break
    return {"value": n / el, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} decode steps of sequence 0 of {case.n_seqs} (append 1 token, decode over "
                      f"{int(case.seq_lens[0])} tokens, W_O) in numpy fp64; BLAS threads use the listed cores"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    case = decode_workload(args)
    st = OracleStep(case, 0)
    for _ in range(max(args.warmup, 3)):
        st.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.step()
    el = time.perf_counter() - t0
    value = args.steps / el
    sample = (f"each step = one decode step (append, decode over {int(case.seq_lens[0])} tokens, W_O) of sequence 0 "
              f"of {case.n_seqs}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_text(case), "batch": case.n_seqs, "ctx": int(np.max(case.seq_lens)),
                   "n_q_heads": case.n_q_heads, "n_kv_heads": case.n_kv_heads, "d_model": case.d_model},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Secondary cases (profiling only)
# ---------------------------------------------------------------------------

def append_chunk_measure(device: str, dense: bool, steps: int, warmup: int, min_s: float = 0.0) -> dict:
    """4,096-token prefill append per sequence: 4 sequences of the 4B-class layer (signed
    Hadamard, clip 0.9), or (dense) of the 8B-class layer (dense R).  Blocks of `steps`
    appends are timed with events on the launching stream and repeated until `min_s`
    seconds have passed; the median block gives the time per append call."""
    import torch
    import int2_kv_cache_gb300 as kvq
    from int2_kv_cache_gb300 import workloads as W
    n_seq = 4
    c = W.gqa8b_32k(n_seqs=n_seq, ctx=4096) if dense else W.long4b_128k(n_seqs=n_seq, ctx=4096)
    t = lambda x, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(x)).to(device).to(dt)
    lay = kvq.make_layout(16, 8, 32, c.num_blocks, c.block_table.shape[1])
    pool = torch.zeros(kvq.kvq_pool_bytes(lay), dtype=torch.uint8, device=device)
    kv = [c.kv(b) for b in range(n_seq)]
    k = t(np.concatenate([x[0] for x in kv]), torch.bfloat16)
    v = t(np.concatenate([x[1] for x in kv]), torch.bfloat16)
    # consecutive appends read different copies of the inputs (3 x 67 MB > the 129 MB L2),
    # so every call streams its K and V from DRAM
    copies = [(k, v)] + [(k.clone(), v.clone()) for _ in range(2)]
    cu = t(np.arange(n_seq + 1) * 4096, torch.int32)
    st = t(np.zeros(n_seq), torch.int32)
    table = t(c.block_table, torch.int32)
    rk, rv = kvq.DeviceRot.from_spec(c.rot_k, device), kvq.DeviceRot.from_spec(c.rot_v, device)
    mu_rot = torch.zeros(8, 128, device=device)

    stream = torch.cuda.current_stream()

    it = [0]

    def step():
        kc, vc = copies[it[0] % len(copies)]
        it[0] += 1
        kvq.kvq_quantize_append(lay, kc, vc, cu, st, table, rk, rv, mu_rot, c.clip_k, c.clip_v, pool)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    blocks = []
    t0 = time.perf_counter()
    while True:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        e1.synchronize()
        blocks.append(e0.elapsed_time(e1) / steps)
        if time.perf_counter() - t0 >= min_s or len(blocks) >= MAX_BLOCKS:
            break
    ms = float(np.median(blocks))
    # algorithmic bytes: bf16 K and V read (2 x 256 B per token-head), 72 B of codes and
    # meta written per token-head, the rotation inputs (signs or dense R) and mu R_K read
    rot_bytes = 2 * 8 * 128 * 4 if not dense else 2 * 8 * 128 * 128 * 4
    bytes_ = n_seq * 4096 * 8 * (2 * 256 + 72) + rot_bytes + 8 * 128 * 4
    peak, kind = peaks()
    achieved = bytes_ / ms / 1e6
    out = {"workload": (f"prefill-chunk quantize-append: {n_seq} sequences x 4,096 new tokens, Hkv 8, d 128, bf16 K/V, "
                        + ("dense expm(A-A^T) rotations, clip 1" if dense else "signed-Hadamard rotations, clip 0.9")
                        + ", 16-token pages"),
           "ms": ms, "tokens": n_seq * 4096, "blocks": len(blocks),
           "l2": "inputs cycled over 3 copies (%.0f MB > 129 MB L2)" % (3 * 2 * k.numel() * 2 / 1e6),
           "roofline": {"kernel": "kvq_quantize_append (prefill chunk)", "bound": "hbm", "achieved": achieved,
                        "peak": peak, "peak_kind": kind, "unit": "GB/s", "frac": achieved / peak,
                        "algorithmic_bytes": bytes_}}
    if dense:
        # the rotation x R_h on the tensor cores: one 128 x 128 x 128 product per (role, head, 128-token
        # tile), done as three exact bf16 limb products of R (bf16 K/V are one limb)
        flops = 2 * 8 * (n_seq * 4096) * 128 * 128 * 2
        out["tensor"] = {"algorithmic_gflop": flops / 1e9, "limb_products": 3,
                         "tflops_algorithmic": flops / ms / 1e9, "tflops_issued": 3 * flops / ms / 1e9}
    return out


def run_append_chunk(args):
    r = append_chunk_measure("cuda:0", args.case == "append_chunk_dense", args.steps, args.warmup)
    print(json.dumps({"case": args.case, **r}), flush=True)


def run_calib(args):
    import torch
    import int2_kv_cache_gb300 as kvq
    from int2_kv_cache_gb300 import workloads as W
    device = "cuda:0"
    cc = W.serve14b_calibration()
    t = lambda x, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(x)).to(device).to(dt)
    bf = torch.bfloat16
    mu = torch.empty(cc.n_kv_heads, 128, device=device)
    kvq.kvq_key_mean(t(cc.k, bf), mu)
    ws = torch.empty(kvq.kvq_calib_workspace_size(cc.n_tok, cc.n_qpos, cc.n_kv_heads, cc.gqa, False),
                     dtype=torch.uint8, device=device)
    nm = torch.empty(len(cc.cands), len(cc.clips), cc.n_kv_heads, dtype=torch.float64, device=device)
    ref = torch.empty(cc.n_kv_heads, dtype=torch.float64, device=device)
    cands = [kvq.DeviceRot.from_spec(x, device) for x in cc.cands]
    q, k, v, w = t(cc.q, bf), t(cc.k, bf), t(cc.v, bf), t(cc.w_o, bf)

    def step():
        kvq.kvq_calib_nmse(q, k, v, w, cands, cc.clips, mu, False, nm, ref, ws)

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    n = max(1, min(args.steps, 3))
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"case": "calib", "ms": e0.elapsed_time(e1) / n, "candidates": len(cc.cands),
                      "clips": len(cc.clips), "heads": cc.n_kv_heads}), flush=True)


def run_report(args):
    """Per-head output-error report on the 14B-class calibration trace: the first two
    dense candidates as R_K and R_V, key centring, Table A's clips 0.96 / 0.92."""
    import torch
    import int2_kv_cache_gb300 as kvq
    from int2_kv_cache_gb300 import workloads as W
    device = "cuda:0"
    cc = W.serve14b_calibration(n_cand=2)
    t = lambda x, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(x)).to(device).to(dt)
    bf = torch.bfloat16
    mu = torch.empty(cc.n_kv_heads, 128, device=device)
    kvq.kvq_key_mean(t(cc.k, bf), mu)
    ws = torch.empty(kvq.kvq_report_workspace_size(cc.n_tok, cc.n_qpos, cc.n_kv_heads, cc.gqa),
                     dtype=torch.uint8, device=device)
    out = torch.empty(5, cc.n_kv_heads, dtype=torch.float64, device=device)
    rk, rv = (kvq.DeviceRot.from_spec(x, device) for x in cc.cands[:2])
    q, k, v, w = t(cc.q, bf), t(cc.k, bf), t(cc.v, bf), t(cc.w_o, bf)

    def step():
        kvq.kvq_head_error_report(q, k, v, w, rk, rv, mu, 0.96, 0.92, out, ws)

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    n = max(1, min(args.steps, 5))
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    print(json.dumps({"case": "report", "ms": e0.elapsed_time(e1) / n, "heads": cc.n_kv_heads, "n_tok": cc.n_tok,
                      "n_qpos": cc.n_qpos, "rms_pct_of_naive": [round(float(x), 2) for x in 100 * np.sqrt(o[0] / o[3])],
                      "key_share": [round(float(x), 3) for x in o[1] / (o[1] + o[2])]}), flush=True)


def run_optr(args):
    """OptR gradient calibration (Algorithm 1) of the 14B-class serving layer's heads:
    each head a 2,560-token training trace and a held-out trace of the same size
    (the last 64 query positions, 4 query heads), d_model 5,120, clips 0.96 / 0.92,
    lambda_K = 1, Adam at 0.02 for --optr-steps steps per phase, selection every 20."""
    import torch
    import int2_kv_cache_gb300 as kvq
    from int2_kv_cache_gb300 import workloads as W
    device = "cuda:0"
    steps = args.optr_steps
    n_tok, n_qpos, gqa, dm = 2560, 64, 4, 5120
    c = W.optr_head(5, n_tok, n_qpos, gqa, dm)
    t32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)
    t64 = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(device)
    q, k, v = c.train
    mu = k.mean(axis=0)
    tr = tuple(t32(x) for x in c.train)
    ho = tuple(t32(x) for x in c.heldout)
    ws = torch.empty(kvq.kvq_optr_workspace_size(n_tok, n_qpos, gqa, n_tok, n_qpos), dtype=torch.uint8, device=device)
    r_k = torch.empty(128, 128, dtype=torch.float64, device=device)
    r_v = torch.empty_like(r_k)
    lk = torch.empty(steps, dtype=torch.float64, device=device)
    lv = torch.empty_like(lk)
    args_ = (tr, ho, t32(c.w_o), t32(mu), t64(c.r_k0), t64(c.r_v0), W.f32(0.96), W.f32(0.92), 1.0, steps,
             W.f32(0.02), 20, r_k, r_v, lk, lv, ws)
    kvq.kvq_optr_calibrate_head(*args_[:9], 2, W.f32(0.02), 20, *args_[12:])  # warm-up (2 steps)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    kvq.kvq_optr_calibrate_head(*args_)
    e1.record()
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    ms = e0.elapsed_time(e1)
    # algorithmic fp64 flops of one loss + gradient evaluation: the exponential and its Frechet
    # derivative (18 + 3 x 17 products of 128 x 128), the effective rows, the causal logits,
    # C = (p^K - p) V, U = C_j M_j and G = U V^T over the pairs, and the backward products
    npairs = n_qpos * gqa
    tok_sum = sum(n_tok - n_qpos + i + 1 for i in range(n_qpos)) * gqa
    mm = 2.0 * 128 ** 3
    pair = 4.0 * 128 * tok_sum + 2.0 * npairs * 128 * 128
    fwd = 18 * mm + 2 * (2.0 * n_tok * 128 * 128) + pair
    bwd = 2.0 * 128 * tok_sum + 2.0 * n_tok * 128 * npairs + 3 * (2.0 * n_tok * 128 * 128) + mm + 3 * 17 * mm
    once = gqa * 2.0 * 128 * 128 * dm + 2 * 2.0 * 128 * tok_sum  # the Gram matrices, both traces' raw logits
    flops = steps * 2 * (fwd + bwd) + once  # both phases (the value phase is cheaper: an upper count)
    peak = 1250.0  # GFLOP/s, GB300 fp64 (nominal)
    print(json.dumps({"case": "optr", "workload": (f"OptR Algorithm 1, one KV head of the 14B-class serving layer: "
                                                   f"{n_tok} tokens, last {n_qpos} positions x {gqa} query heads, "
                                                   f"d_model {dm}, {steps} + {steps} Adam steps, held-out selection"),
                      "ms_per_head": ms, "s_per_layer_10_heads": 10 * ms / 1e3,
                      "final_losses": [float(lk[-1]), float(lv[-1])],
                      "roofline": {"bound": "alu (fp64)", "achieved_gflops": flops / ms / 1e6, "peak": peak,
                                   "unit": "GFLOP/s", "frac": flops / ms / 1e6 / peak, "flops": flops}}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.case in ("append_chunk", "append_chunk_dense"):
        run_append_chunk(args)
    elif args.case == "report":
        run_report(args)
    elif args.case == "calib":
        run_calib(args)
    elif args.case == "optr":
        run_optr(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
