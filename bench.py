"""Benchmark of the sink + low-rank decode path on B300.

One "step" = one decode step of every head of the workload (fused read-out +
factored update), with the recompression back to rank r that runs after
every T-th step amortised over its T steps, so the figure is whole-job
head-steps/s: value = heads / (mean decode time + mean recompression time / T).
The default workload is the largest one that fits one GPU, the serving-scale
Gated DeltaNet batch (589,824 heads of 128 x 128, ragged ranks 16/32/48).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  Inputs of every step are generated on the
device before the timed region and stay resident in HBM; L2 is flushed
(a 256 MiB write followed by a 256 MiB read) before every timed step, and each timed step is bracketed
by CUDA events on the launching stream.  ``--impl reference`` times the CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = 'factored-state decode head-steps/s and HBM GB/s vs 8 TB/s; dense-state ratio'
UNIT = 'head-steps/s'
DEFAULT_WORKLOAD = 'gdn_serving_b512_l36_h32_ragged'
FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument('--gpus', type=int, default=1)
    ap.add_argument('--steps', type=int, default=32)
    ap.add_argument('--warmup', type=int, default=4)
    ap.add_argument('--workload', default=DEFAULT_WORKLOAD)
    ap.add_argument('--impl', default='seed', choices=['seed', 'reference'])
    ap.add_argument('--cpu-seconds', type=float, default=12.0, help='budget of the CPU-oracle sample')
    ap.add_argument('--warm-seconds', type=float, default=0.5,
                    help='keep warming up (after the W steps) until this much time has passed')
    ap.add_argument('--no-dense', action='store_true')
    ap.add_argument('--no-e2e', action='store_true')
    ap.add_argument('--no-cpu', action='store_true')
    ap.add_argument('--recompress', default='phases', choices=['phases', 'single'],
                    help='three-phase recompression over a workspace, or the single kernel')
    ap.add_argument('--ws-heads', type=int, default=0,
                    help='heads per recompression workspace chunk (default: the library default)')
    ap.add_argument('--requests', type=int, default=0,
                    help='run the workload with this many requests instead of its own count '
                         '(the same shapes on a smaller batch, for profiling captures)')
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get('WORLD_SIZE', '1'))
    rank = int(os.environ.get('RANK', '0'))
    local = int(os.environ.get('LOCAL_RANK', '0'))
    return ws, rank, local


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------

def oracle_sample(w, seconds: float, n_sample: int = 64):
    """Time the CPU oracle on a sample of the workload's heads: decode steps from a
    rank-r state with recompression every T steps, until ``seconds`` have passed."""
    import numpy as np
    import oracle
    import synth
    rng = np.random.default_rng(0)
    heads = rng.choice(w.n_heads, size=min(n_sample, w.n_heads), replace=False)
    ranks = synth.head_ranks(w, heads)
    growth = w.growth
    states = []
    for i, h in enumerate(heads):
        d = synth.head_dir(w, h)
        vbar = synth.sink_directions(w, [d])[0]
        r = int(ranks[i])
        raw = synth.random_factored_state(w.seed + 7, 1, w.d_k, w.d_v, [r], r + growth * w.T, w.variant)
        st = oracle.FactoredState(a=raw['a'][0], U=raw['U'][0, :r].T, W=raw['W'][0, :r].T, vbar=vbar)
        if w.variant == 'kda':
            st.D = np.ones(w.d_k)
        else:
            st.scale = np.ones(r)
        A = float(synth.mamba2_A(w, [d])[0]) if w.variant == 'mamba2' else None
        states.append((st, A, r))
    done = 0
    t0 = time.perf_counter()
    step = 0
    while True:
        toks = synth.decode_inputs(w, step % w.steps, heads)
        for i in range(len(heads)):
            st, A, r = states[i]
            st, _ = oracle.factored_step(w.variant, st, {k: v[i] for k, v in toks.items()}, A)
            if (step + 1) % w.T == 0:
                st, _ = oracle.recompress(st, r)
            states[i] = (st, A, r)
        done += len(heads)
        step += 1
        el = time.perf_counter() - t0
        if el >= seconds and step % w.T == 0:
            break
    return dict(value=done / el, unit=UNIT, cores=1, kind='oracle',
                sample=f'{len(heads)} sampled heads x {step} decode steps (recompression every {w.T}), '
                       f'float64 numpy, one thread, {el:.1f} s')


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    os.environ.setdefault('OPENBLAS_NUM_THREADS', '1')
    steps = []
    budget = max(0.02, min(1.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(max(0, args.warmup)):
        oracle_sample(w, budget, n_sample=16)
    for _ in range(args.steps):
        steps.append(oracle_sample(w, budget, n_sample=16))
    value = statistics.mean(s['value'] for s in steps)
    cb = dict(steps[-1])
    cb['value'] = value
    out = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=ws, steps=args.steps, warmup=args.warmup,
               ms_per_step=1e3 * w.n_heads / value, higher_is_better=True, scaling='weak',
               vs_baseline=None, dtype='f64', data='synthetic', impl='reference',
               config=dict(workload=w.name, heads=w.n_heads, d_k=w.d_k, d_v=w.d_v, r=w.r_max, T=w.T,
                           factor_dtype='f64'),
               cpu_baseline=cb, e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

class ClockSampler:
    """Samples the SM clock and the clock-event reasons while running.

    Read-only NVML queries through ctypes on libnvidia-ml (no Python NVML
    package needed); nothing is set.
    """
    REASONS = {0x1: 'gpu_idle', 0x2: 'applications_clocks_setting', 0x4: 'sw_power_cap',
               0x8: 'hw_slowdown', 0x10: 'sync_boost', 0x20: 'sw_thermal_slowdown',
               0x40: 'hw_thermal_slowdown', 0x80: 'hw_power_brake_slowdown', 0x100: 'display_clock_setting'}
    NVML_CLOCK_SM = 1

    def __init__(self, index: int, period: float = 0.002):
        import ctypes
        self.samples = []
        self.period = period
        self._stop = threading.Event()
        self.ok = False
        self.why = ''
        self.max_mhz = None
        try:
            nv = ctypes.CDLL('libnvidia-ml.so.1')
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError('nvmlInit_v2 failed')
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                raise RuntimeError('no NVML handle')
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.reason_fn = getattr(nv, 'nvmlDeviceGetCurrentClocksEventReasons', None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self.ct = nv, h, ctypes
            self.ok = True
        except Exception as e:
            self.why = f'{type(e).__name__}: {e}'

    def _run(self):
        ct = self.ct
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            a = self.nv.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ct.byref(mhz))
            b = self.reason_fn(self.h, ct.byref(rs))
            if a == 0 and b == 0:
                self.samples.append((time.perf_counter(), mhz.value, rs.value))
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self.ok:
            self.t.join()

    def summary(self, t0: float, t1: float):
        if not self.ok:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=['nvml unavailable: ' + self.why])
        inside = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples[-5:]
        mhz = statistics.median(s[1] for s in inside) if inside else None
        bits = 0
        for s in inside:
            bits |= s[2]
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b)
        return dict(sm_mhz=mhz, sm_max_mhz=self.max_mhz, reasons=reasons, samples=len(inside))


def measured_peaks():
    p = os.path.join(ROOT, 'MEASURED_PEAKS.json')
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d['hbm_gbs'], src='measured')
    return dict(hbm_gbs=6400.0, src='fallback')


# Sources whose compiled kernels a committed ncu summary describes; a summary
# counts only while the hash of these files is the one it records.
PROFILE_SOURCES = {
    'decode': ['decode_mma.cu', 'common.cuh'],
    # 16-bit factors: Cholesky of the value-side Gram matrix (gram_phase, evd_phase, gram_rebuild)
    'recompress': ['recompress_gram.cu', 'evd_warp.cuh', 'svd_warp.cuh', 'recompress_core.cuh', 'common.cuh'],
    # 32-bit factors: QR of both factors (qr_phase, svd_phase, rebuild_phase)
    'recompress_f32': ['recompress_split.cu', 'qr_registers.cuh', 'svd_warp.cuh', 'recompress_core.cuh',
                       'common.cuh'],
}


def source_hash(kind: str) -> str:
    h = hashlib.sha256()
    for f in PROFILE_SOURCES[kind]:
        with open(os.path.join(ROOT, 'rank_state_compression_head_b300', 'csrc', f), 'rb') as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_record(kind: str, workload: str):
    """Key/value lines of profiles/ncu_<kind>_<workload>.md if its sources are unchanged, else None."""
    path = os.path.join(ROOT, 'profiles', f'ncu_{kind}_{workload}.md')
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if ':' in line and line.startswith('- '):
                k, v = line[2:].split(':', 1)
                rec[k.strip()] = v.strip()
    if rec.get('source_sha256_16') != source_hash(kind):
        return None
    return rec


def run_gpu(args, w):
    import numpy as np
    import torch
    import torch.distributed as dist
    from rank_state_compression_head_b300 import accounting as acc
    from rank_state_compression_head_b300 import sharding
    from rank_state_compression_head_b300.workload import DEFAULT_WS_HEADS, DeviceRun

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group('nccl')
    w = sharding.shard(w, rank, ws)  # each rank: its own batch of requests of the workload's shapes
    torch.cuda.set_device(local)
    dev = torch.device('cuda', local)
    stream = torch.cuda.current_stream()
    T = w.T
    K, W_ = args.steps, max(3, args.warmup)
    total_steps = K + W_

    # ---- setup: constants, prefill, compression, inputs of every step -----------------
    ws_heads = (args.ws_heads or DEFAULT_WS_HEADS) if args.recompress == 'phases' else 0
    run = DeviceRun(w, device=dev, steps_buffered=total_steps, ws_heads=ws_heads)
    rec_launches = run.recompress_launches()
    # setup, timed once (not part of the decode metric): dense prefill and compression
    ev_setup = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev_setup[0].record(stream)
    S_dense = run.prefill()
    ev_setup[1].record(stream)
    run.compress(S_dense)
    ev_setup[2].record(stream)
    for t in range(total_steps):
        run.gen_inputs(t % w.steps, slot=t)
    torch.cuda.synchronize()
    ranks_host = run.ranks.cpu().numpy().astype(np.int64)
    flush_w = torch.empty(FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    flush_r = torch.ones(FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    flush_out = torch.empty((), device=dev, dtype=torch.float32)

    def l2_flush():
        # write a buffer larger than L2, then read another one: L2 ends up holding clean,
        # unrelated lines, so the timed step neither hits its own data nor pays for
        # writing back the flush's dirty lines
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_out)

    sweeps = torch.zeros(run.H, device=dev, dtype=torch.int32)

    uniq, counts = np.unique(ranks_host, return_counts=True)

    def launch_bytes(s_before):  # algorithmic bytes of one decode launch at this point of the interval
        return sum(int(c) * acc.decode_bytes(w.variant, w.d_k, w.d_v, int(r) + w.growth * s_before,
                                              w.factor_dtype) for r, c in zip(uniq, counts))

    bytes_at = [launch_bytes(s) for s in range(T)]
    cols_at = [int(ranks_host.sum()) + run.H * w.growth * s for s in range(T)]

    # ---- warm-up (brings clocks up, fills caches and code) ---------------------------
    t_end = time.perf_counter() + args.warm_seconds
    t = 0
    while t < W_ or time.perf_counter() < t_end:
        l2_flush()
        run.decode(slot=t % total_steps)
        if run.state.steps_since_compress == T:
            run.recompress()
        t += 1
        if t > 20000:
            break
    # continue the schedule from a compression boundary
    if run.state.steps_since_compress:
        run.recompress()
    torch.cuda.synchronize()

    # ---- timed region ------------------------------------------------------------------
    # Arguments of every call are built before timing so that the host issues each
    # step in a few microseconds and the GPU queue never drains inside a step.
    import ctypes
    from rank_state_compression_head_b300 import _lib
    sptr = stream.cuda_stream
    st_ref = ctypes.byref(run.state.st)
    A_ptr = run.A.data_ptr() if run.A is not None else None
    dec_args = [(st_ref, run.q[W_ + i].data_ptr(), run.k[W_ + i].data_ptr(), run.v[W_ + i].data_ptr(),
                 run.gate[W_ + i].data_ptr(), run.beta[W_ + i].data_ptr(), A_ptr, run.o.data_ptr(), sptr)
                for i in range(K)]
    if run.ws is not None:
        rec_fn = _lib.seed_recompress_ws
        rec_args = (st_ref, run.trunc.data_ptr(), sweeps.data_ptr(), run.ws.data_ptr(), run.ws_bytes, sptr)
    else:
        rec_fn = _lib.seed_recompress_ex
        rec_args = (st_ref, run.trunc.data_ptr(), sweeps.data_ptr(), sptr)
    dec_fn = _lib.seed_decode_step
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    rec_steps = []
    bytes_decode = 0
    m_sum = 0
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        c0 = time.perf_counter()
        for i in range(K):
            l2_flush()
            s_before = run.state.steps_since_compress
            m_sum += cols_at[s_before]
            bytes_decode += bytes_at[s_before]
            ev[i][0].record(stream)
            rc = dec_fn(*dec_args[i])
            ev[i][1].record(stream)
            if run.state.steps_since_compress == T:
                rc |= rec_fn(*rec_args)
                rec_steps.append(i)
            ev[i][2].record(stream)
            if rc:
                raise RuntimeError(f'library call failed with status {rc}')
        torch.cuda.synchronize()
        c1 = time.perf_counter()
        # Fewer than T timed steps hold no recompression: run the schedule on (untimed)
        # to the next boundary and time that recompression alone, the same way.
        if not rec_steps:
            while run.state.steps_since_compress < T:
                run.decode(slot=(W_ + K) % total_steps)
            l2_flush()
            ev_extra = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev_extra[0].record(stream)
            rc = rec_fn(*rec_args)
            ev_extra[1].record(stream)
            if rc:
                raise RuntimeError(f'library call failed with status {rc}')
            torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    dec_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    rec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in rec_steps] or [ev_extra[0].elapsed_time(ev_extra[1])]
    # Whole-job time of one step: its decode plus 1/T of a recompression (one runs
    # after every T-th step), so any K gives the long-run rate.
    step_ms_amortised = statistics.mean(dec_ms) + statistics.mean(rec_ms) / T
    total_ms = sharding.max_over_ranks(step_ms_amortised * K, device=dev)
    heads_all = sharding.job_heads(run.H, ws)
    value = heads_all * K / (total_ms / 1e3)
    clocks = clk.summary(c0, c1)
    sw = sweeps.cpu().numpy()

    # ---- roofline of each kernel ---------------------------------------------------------
    peaks = measured_peaks()
    dec_avg_ms = statistics.mean(dec_ms)
    dec_gbs = (bytes_decode / K) / (dec_avg_ms / 1e3) / 1e9
    m_rec = ranks_host + w.growth * T
    rec_flops = float(sum(acc.recompress_flops(w.d_k, w.d_v, int(mm), int(rr), float(max(s, 1)))
                          for mm, rr, s in zip(m_rec, ranks_host, sw)))
    rec_avg_ms = statistics.mean(rec_ms) if rec_ms else float('nan')
    fp32_peak = 148 * 128 * 2 * (clocks['sm_max_mhz'] or 2032) * 1e6 / 1e12  # TFLOP/s, FFMA issue rate
    rec_tflops = rec_flops / (rec_avg_ms / 1e3) / 1e12 if rec_ms else None
    dec_total, rec_total = statistics.mean(dec_ms) * K, statistics.mean(rec_ms) * K / T  # amortised
    # DRAM bytes per launch from the committed ncu captures: the decode capture is
    # one launch at a known column count, scaled to this run's mean algorithmic
    # bytes; the recompression capture covers its three kernels at m = r + growth*T.
    traffic, rec_traffic = None, None
    prof = profiled_record('decode', w.name)
    if prof is not None:
        try:
            traffic = round(float(prof['traffic_bytes_per_launch']) * (bytes_decode / K)
                            / float(prof['algorithmic_bytes_per_launch']))
        except (KeyError, ValueError, ZeroDivisionError):
            traffic = None
    prof = profiled_record('recompress' if w.factor_dtype != 'f32' else 'recompress_f32', w.name)
    if prof is not None and run.ws is not None:
        try:
            rec_traffic = round(float(prof['traffic_bytes_per_launch']))
        except (KeyError, ValueError):
            rec_traffic = None
    roof_dec = dict(kernel='decode_mma_kernel' if w.factor_dtype != 'f32' else 'decode_kernel', bound='hbm',
                    achieved=round(dec_gbs, 1),
                    peak=peaks['hbm_gbs'], unit='GB/s', frac=round(dec_gbs / peaks['hbm_gbs'], 4),
                    traffic=traffic, peak_src=peaks['src'],
                    algorithmic_bytes_per_launch=round(bytes_decode / K),
                    avg_launch_us=round(dec_avg_ms * 1e3, 3))
    if run.ws is None:
        rec_kernels = 'recompress_kernel'
    elif w.factor_dtype == 'f32':
        rec_kernels = 'qr_phase + svd_phase + rebuild_phase'
    else:
        listed = run.state.ranks is not None and run.state.head_order is None  # class lists on the device
        rec_kernels = ('gram_classify + ' if listed else '') + 'gram_phase + evd_phase + gram_rebuild'
    roof_rec = dict(kernel=f'{rec_kernels} (recompress)', bound='alu', achieved=rec_tflops and round(rec_tflops, 3),
                    peak=round(fp32_peak, 1), unit='TFLOP/s',
                    frac=rec_tflops and round(rec_tflops / fp32_peak, 4), traffic=rec_traffic,
                    peak_src='148 SMs x 128 FP32 lanes x 2 FLOP x max SM clock',
                    algorithmic_flops_per_launch=round(rec_flops), avg_launch_us=round(rec_avg_ms * 1e3, 1),
                    jacobi_sweeps_mean=float(np.mean(sw)), jacobi_sweeps_max=int(np.max(sw)))
    dominant = roof_dec if dec_total >= rec_total else roof_rec

    out = dict(metric=METRIC, value=round(value), unit=UNIT, n_gpus=ws, steps=K, warmup=W_,
               ms_per_step=round(total_ms / K, 5), higher_is_better=True, scaling='weak',
               vs_baseline=None, dtype='f32', data='synthetic',
               config=dict(workload=w.name, heads_per_gpu=run.H, d_k=w.d_k, d_v=w.d_v, r=w.r_max,
                           T=w.T, factor_dtype=w.factor_dtype, variant=w.variant,
                           l2='flushed before every timed step (256 MiB write then 256 MiB read, untimed)',
                           parallelism=f'heads sharded over {ws} rank(s), one batch of requests each'),
               roofline=dominant, gpu_launches=K * run.decode_launches() + rec_launches * len(rec_ms),
               clocks=clocks)
    out['config']['recompression'] = (f'after every {T}th step, amortised: ms_per_step = mean decode + '
                                      f'mean recompression / {T} ({len(rec_ms)} recompression(s) timed)')
    out['decode'] = dict(head_steps_per_s=round(heads_all * K / (dec_total / 1e3)),
                         us_per_step=round(dec_avg_ms * 1e3, 3), gbs=round(dec_gbs, 1),
                         frac_of_measured_hbm=round(dec_gbs / peaks['hbm_gbs'], 4),
                         frac_of_8tbs=round(dec_gbs / 8000.0, 4),
                         bytes_per_head_step=round(bytes_decode / K / run.H, 1),
                         mean_columns=round(m_sum / K / run.H, 2))
    out['recompress'] = roof_rec
    out['setup'] = dict(dense_prefill_ms=round(ev_setup[0].elapsed_time(ev_setup[1]), 3),
                        compress_dense_ms=round(ev_setup[1].elapsed_time(ev_setup[2]), 3),
                        compress_dense_us_per_head=round(ev_setup[1].elapsed_time(ev_setup[2]) * 1e3 / run.H, 3))
    out['time_share'] = dict(decode=round(dec_total / total_ms, 4), recompress=round(rec_total / total_ms, 4))

    # ---- dense-state comparator ----------------------------------------------------------
    if not args.no_dense:
        o_d = torch.empty_like(run.o)
        for t in range(W_):
            run.dense_step(S_dense, slot=t, o=o_d)
        dev_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        torch.cuda.synchronize()
        dn_fn = _lib.seed_dense_decode_step
        dn_args = [(run.variant, run.H, w.d_k, w.d_v, S_dense.data_ptr(), run.q[W_ + i].data_ptr(),
                    run.k[W_ + i].data_ptr(), run.v[W_ + i].data_ptr(), run.gate[W_ + i].data_ptr(),
                    run.beta[W_ + i].data_ptr(), A_ptr, run.vbar_index.data_ptr(), o_d.data_ptr(), sptr)
                   for i in range(K)]
        for i in range(K):
            l2_flush()
            dev_ev[i][0].record(stream)
            if dn_fn(*dn_args[i]):
                raise RuntimeError('dense step failed')
            dev_ev[i][1].record(stream)
        torch.cuda.synchronize()
        dms = statistics.mean(dev_ev[i][0].elapsed_time(dev_ev[i][1]) for i in range(K))
        dbytes = run.H * acc.dense_decode_bytes(w.variant, w.d_k, w.d_v)
        out['dense'] = dict(us_per_step=round(dms * 1e3, 3), head_steps_per_s=round(run.H * ws / (dms / 1e3)),
                            gbs=round(dbytes / (dms / 1e3) / 1e9, 1),
                            bytes_per_head_step=acc.dense_decode_bytes(w.variant, w.d_k, w.d_v),
                            bytes_ratio_dense_over_factored=round(dbytes / (bytes_decode / K), 3),
                            time_ratio_dense_over_factored_decode=round(dms / dec_avg_ms, 3),
                            time_ratio_dense_over_factored_with_recompress=round(dms / (total_ms / K), 3))

    # ---- end to end through host buffers -------------------------------------------------
    # Every step's inputs (q, k, v, gate, beta packed in one pinned buffer) go host ->
    # device and its output device -> host inside the timed region.  Copies run on
    # their own streams into two device slots, so that the upload of step t+1 and
    # the download of step t-1 overlap the kernels of step t; events keep each slot
    # from being overwritten before it has been consumed.  The pinned host side is a
    # ring of a few step-sized slots (the serving workload moves ~0.9 GB in per step).
    # One untimed interval of T steps warms the copy engines and the recompression up;
    # the timed run covers whole intervals (K rounded up to a multiple of T), so each
    # recompression is counted once per T steps.
    if not args.no_e2e:
        H = run.H
        segs = [run.q[0].numel(), run.k[0].numel(), run.v[0].numel(), run.gate[0].numel(), run.beta[0].numel()]
        offs = np.concatenate([[0], np.cumsum(segs)]).astype(np.int64)
        n_in = int(offs[-1])
        assert all(int(o) % 4 == 0 for o in offs)          # 16-byte aligned segments
        K_e2e = -(-K // T) * T
        W_e2e = max(T, W_)
        n_host = min(4, total_steps)
        hin = torch.empty(n_host, n_in, pin_memory=True)
        for j, src in enumerate((run.q, run.k, run.v, run.gate, run.beta)):
            hin[:, offs[j]:offs[j + 1]].copy_(src[:n_host].reshape(n_host, -1))
        hout = torch.empty(n_host, *run.o.shape, pin_memory=True)
        # device slots for the steps' inputs and outputs: the uploads run up to
        # n_dev - 1 steps ahead of the compute, so the host link keeps streaming while
        # a recompression runs
        n_dev = 4
        din = [torch.empty(n_in, device=dev) for _ in range(n_dev)]
        dout = [torch.empty_like(run.o) for _ in range(n_dev)]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        # Raw runtime calls keep the host's issue cost per step to a few microseconds,
        # well under the copy time, so the host runs ahead of the GPU.
        rt = ctypes.CDLL('libcudart.so.13')
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        rt.cudaMemcpyAsync.argtypes = [vp, vp, sz, ctypes.c_int, vp]
        rt.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
        rt.cudaEventRecord.argtypes = [vp, vp]
        rt.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
        rt.cudaEventDestroy.argtypes = [vp]

        def new_events(n):
            out_ = []
            for _ in range(n):
                e = vp()
                if rt.cudaEventCreateWithFlags(ctypes.byref(e), 2):  # cudaEventDisableTiming
                    raise RuntimeError('cudaEventCreateWithFlags failed')
                out_.append(e)
            return out_
        n_ev = max(K_e2e, W_e2e)
        h2d_done, comp_done, d2h_done = new_events(n_ev), new_events(n_ev), new_events(n_ev)
        h2d = n_in * 4
        d2h = run.o.numel() * 4
        s_up, s_down = vp(up.cuda_stream), vp(down.cuda_stream)
        s_comp = vp(sptr)
        hin_p = [hin[i].data_ptr() for i in range(n_host)]
        hout_p = [hout[i].data_ptr() for i in range(n_host)]
        din_p = [t.data_ptr() for t in din]
        dout_p = [t.data_ptr() for t in dout]
        in_args = [[dp + int(o) * 4 for o in offs[:5]] for dp in din_p]

        def e2e_loop(n):
            """n steps from a compression boundary; the last ends on one when T | n."""
            def upload(i):
                if i >= n_dev:
                    rt.cudaStreamWaitEvent(s_up, comp_done[i - n_dev], 0)  # slot consumed by step i - n_dev
                rc_ = rt.cudaMemcpyAsync(din_p[i % n_dev], hin_p[i % n_host], h2d, 1, s_up)
                rt.cudaEventRecord(h2d_done[i], s_up)
                return rc_

            up.wait_stream(stream)
            down.wait_stream(stream)
            rc = 0
            for i in range(min(n_dev - 1, n)):
                rc |= upload(i)
            for i in range(n):
                slot = i % n_dev
                if i + n_dev - 1 < n:
                    rc |= upload(i + n_dev - 1)
                rt.cudaStreamWaitEvent(s_comp, h2d_done[i], 0)
                if i >= n_dev:
                    rt.cudaStreamWaitEvent(s_comp, d2h_done[i - n_dev], 0)  # output slot read back
                a_ = in_args[slot]
                rc |= dec_fn(st_ref, a_[0], a_[1], a_[2], a_[3], a_[4], A_ptr, dout_p[slot], sptr)
                if run.state.steps_since_compress == T:
                    rc |= rec_fn(*rec_args)
                rt.cudaEventRecord(comp_done[i], s_comp)
                rt.cudaStreamWaitEvent(s_down, comp_done[i], 0)
                rc |= rt.cudaMemcpyAsync(hout_p[i % n_host], dout_p[slot], d2h, 2, s_down)
                rt.cudaEventRecord(d2h_done[i], s_down)
            if rc:
                raise RuntimeError(f'end-to-end loop: a call failed (status {rc})')
            rt.cudaStreamWaitEvent(s_comp, d2h_done[n - 1], 0)

        torch.cuda.synchronize()
        if run.state.steps_since_compress:
            run.recompress()
        e2e_loop(W_e2e)                                   # untimed warm-up interval
        torch.cuda.synchronize()
        if run.state.steps_since_compress:
            run.recompress()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_loop(K_e2e)
        e1.record(stream)
        torch.cuda.synchronize()
        for e in h2d_done + comp_done + d2h_done:
            rt.cudaEventDestroy(e)
        e2e_ms = e0.elapsed_time(e1)
        e2e_ms = sharding.max_over_ranks(e2e_ms, device=dev)
        out['e2e'] = dict(value=round(heads_all * K_e2e / (e2e_ms / 1e3)), unit=UNIT,
                          h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                          ms_per_step=round(e2e_ms / K_e2e, 5), steps=K_e2e, warmup_steps=W_e2e,
                          host_slots=n_host)

    # ---- CPU oracle baseline (rank 0, N = 1) --------------------------------------------
    if rank == 0 and ws == 1 and not args.no_cpu:
        out['cpu_baseline'] = oracle_sample(w, args.cpu_seconds)
    if sharding.reports(rank):
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    import synth
    if args.workload not in synth.WORKLOADS:
        raise SystemExit(f'unknown workload {args.workload}; one of {sorted(synth.WORKLOADS)}')
    w = synth.WORKLOADS[args.workload]
    if args.requests > 0:
        w = w.with_(n_req=args.requests)
    if args.impl == 'reference':
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == '__main__':
    main()
