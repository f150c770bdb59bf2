"""Benchmark: batch-size-1 greedy decode of a random-init Llama-2-7B-shaped
model (32 layers, d 4096, 32 heads x 128, SwiGLU 11008, vocab 32000, RMSNorm
eps 1e-5, RoPE theta 1e4; 5-token random prompt, then greedy tokens; KV cache
bf16 up to 2048), with int4-G32 weight-only weights as the headline and bf16 /
int8 measured in the same run (the gpt-fast README's "Benchmarks" table:
tokens/s at batch size 1, and the bandwidth those tokens imply).

One step = one decode token = one launch of the persistent engine, which runs
every layer.  `value` is tokens/s with the model resident in HBM (the timed
loop feeds each step's argmax back as the next token on the device); `e2e`
times the same loop through the C-ABI with the token copied in from pinned
host memory and the argmax read back every step.  The model (4.1-13.5 GB) is
far larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--dtype int4|int8|bf16]
                  [--impl ours|reference] [--workload llama2-7b|llama3.1-8b|mixtral-8x7b]
                  [--ctx L1,L2,...] [--verify-k K]

--ctx times the decode from contexts of L positions written straight into the
KV cache (seeded bf16 N(0, 1) rows; the Llama-3.1-8B sweep uses 128, 1024 and
8192), --verify-k adds speculative-verification passes of K draft tokens after
the decode measurement (drafts = the model's own greedy continuation, all
accepted, and uniform random drafts, about none accepted).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PUBLISHED_TOKS = {  # gpt-fast README "Benchmarks", 1x A100-80GB at 330 W (context)
    ("llama2-7b", "bf16"): 104.9, ("llama2-7b", "int8"): 155.58, ("llama2-7b", "int4"): 196.80,
    ("llama3.1-8b", "bf16"): 93.89, ("llama3.1-8b", "int8"): 137.64,
}
METRIC = "bs=1 decode tokens/s and achieved HBM GB/s vs GB300 peak (bf16/int8/int4-G32)"
N_PROMPT = 5


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--dtype", default="int4", choices=["int4", "int8", "bf16"])
    ap.add_argument("--workload", default="llama2-7b",
                    choices=["llama2-7b", "llama3.1-8b", "mixtral-8x7b", "gemv-set", "gemv"])
    ap.add_argument("--ctx", default="", help="comma-separated context lengths written into the KV cache")
    ap.add_argument("--verify-k", type=int, default=0, help="also time verification passes of k drafts")
    ap.add_argument("--speculate", type=int, default=0,
                    help="also time speculative generation with k drafts per round (target --spec-target, "
                         "draft --spec-draft copies of the same model) against plain greedy generation")
    ap.add_argument("--spec-target", default="bf16", choices=["int4", "int8", "bf16"])
    ap.add_argument("--spec-draft", default="int4", choices=["int4", "int8", "bf16"])
    ap.add_argument("--spec-tokens", type=int, default=100)
    ap.add_argument("--prefill", action="store_true",
                    help="also time the 5-token prompt as one gf_prefill pass against 5 decode steps")
    ap.add_argument("--only-headline", action="store_true", help="skip the other two weight dtypes")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--group", type=int, default=32, choices=[32, 64, 128], help="int4 group size along K")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="use only the first L layers (profiling runs)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x, world, device=None):
    """x reduced with MAX over the ranks of the default process group (the
    slowest replica's time decides a multi-GPU number); x itself on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- clocks -----
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
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
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def measured_traffic(workload, dtype):
    """DRAM bytes per k_engine launch from a committed ncu capture
    (profiles/traffic.json), or None when absent, for another workload, or
    taken on a different engine source than the one built now."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for name in ("engine.cu", "gf_internal.cuh"):  # the sources of k_engine
        with open(os.path.join(ROOT, "weight_only_quantized_bs_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    sha = h.hexdigest()[:16]
    r = rec.get("%s/%s" % (workload, dtype))
    if not r or r.get("engine_sha") != sha:
        return None
    return r["bytes_per_launch"]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------ CPU baseline -----
class OracleStream:
    """The oracle as it stands, on one host core, decoding a stream of tokens
    at positions p0, p0 + 1, ... in stages: stage s of a token is layer s
    (s < n_layers) or the final RMSNorm + lm_head (s == n_layers), in that
    order, each on the previous stage's output, so that n_layers + 1
    consecutive stages are one whole token.  The cache rows 0..p0-1 of every
    layer hold seeded bf16 N(0, 1) K and V rows (the context the GPU arm has
    reached at p0).  Building and quantising the layers (`layers_needed` of
    them, in order) happens before any stage and is not timed."""

    def __init__(self, cfg, dtype, seed, p0, layers_needed):
        import oracle
        from synth import models
        self.cfg, self.p0 = cfg, p0
        self.wc = models.WeightCache(cfg, seed=seed, keep=False)
        self.om = oracle.OracleModel(cfg, dtype, self.wc, tmax=p0 + 64, keep=True)
        for l in range(min(layers_needed, cfg["n_layers"])):
            self.om._layer(l)
            if p0 > 0:
                k, v = models.kv_prefill(cfg, seed, l, p0)
                self.om.K[l][:, :p0, :] = oracle.bf16_to_double(k)
                self.om.V[l][:, :p0, :] = oracle.bf16_to_double(v)
        self.tokens = models.prompt(cfg, seed, 64)
        self.n_stages = cfg["n_layers"] + 1
        self.i = 0
        self.x = None

    def stage(self):
        """Runs the next stage; returns its seconds (the lm_head stage's
        logits are kept in self.logits)."""
        import numpy as np
        import oracle
        cfg, om = self.cfg, self.om
        j, s = divmod(self.i, self.n_stages)
        pos = self.p0 + j
        if s == 0:
            self.x = oracle.bf16_to_double(om.embed[[int(self.tokens[j % len(self.tokens)])]])
        t0 = time.perf_counter()
        if s < cfg["n_layers"]:
            self.x = om.layer_forward(s, self.x, pos)
        else:
            self.logits = om.lm_head(np.stack([oracle.rmsnorm(self.x[0], self.wc.glob["g_final"], cfg["eps"])]))[0]
        dt = time.perf_counter() - t0
        self.i += 1
        return dt


def bench_config(args, cfg, tmax, p_first, ctxs):
    """The `config` object of both arms' JSON line (identical for one command)."""
    c = {"workload": "%s-shaped greedy decode, %s weights" % (args.workload, args.dtype),
         "shapes": args.workload, "n_layers": cfg["n_layers"],
         "weights": args.dtype + ("-g%d" % args.group if args.dtype == "int4" else ""),
         "batch": 1, "prompt": 1 if ctxs else N_PROMPT, "tmax": tmax,
         "positions": [p_first, p_first + args.steps],
         "parallelism": "replicas" if args.gpus > 1 else "single",
         "l2": "no flush: every step streams the whole model (GBs), far above the 129 MB L2"}
    if ctxs:
        c["contexts"] = ctxs
    return c


def bench_positions(args):
    """(tmax, first timed position, contexts) of a command line."""
    ctxs = [int(c) for c in args.ctx.split(",") if c]
    tmax = 2048 if not ctxs else max(ctxs) + max(args.warmup, N_PROMPT) + args.steps + 8
    p_first = ctxs[0] + args.warmup if ctxs else max(args.warmup, N_PROMPT)
    return tmax, p_first, ctxs


# ------------------------------------------------- byte accounting -----
def decode_bytes(cfg, weight_bytes, p0, steps):
    """Algorithmic bytes of `steps` decode tokens at positions p0 .. p0 +
    steps - 1: per token the model's streamed weight bytes (gf_model_weight_bytes:
    linear weights incl. lm_head, scales, norm gains, one embedding row) plus
    the bf16 K and V rows 0..pos of every layer read and the row at pos
    written."""
    row = 2 * cfg["n_layers"] * cfg["n_kv_heads"] * cfg["head_dim"] * 2  # K and V of one position
    return weight_bytes * steps + sum(row * (p + 1) + row for p in range(p0, p0 + steps))


# ------------------------------------------------- decode variants -----
class _DevPtr:
    """A device address where the binding expects a tensor."""

    def __init__(self, p):
        self.p = p

    def data_ptr(self):
        return self.p


def fill_context(gf, kv, cfg, seed, ctx, tmax, dev):
    """Writes a context of ctx positions (seeded bf16 N(0, 1) K and V rows)
    straight into every layer's KV cache, [kv head][tmax][head_dim] per layer."""
    import numpy as np
    import torch
    from synth import models
    kp, vp = kv.cache_ptrs()
    Hkv, hd = cfg["n_kv_heads"], cfg["head_dim"]
    layer_bytes = Hkv * tmax * hd * 2
    for l in range(cfg["n_layers"]):
        k, v = models.kv_prefill(cfg, seed, l, ctx)
        for src, base in ((k, kp), (v, vp)):
            full = np.zeros((Hkv, tmax, hd), dtype=np.uint16)
            full[:, :ctx, :] = src
            t = torch.from_numpy(full.view(np.int16)).to(dev)
            gf.copy_ceiling(t, _DevPtr(base + l * layer_bytes), layer_bytes)
    torch.cuda.synchronize()


def measure_verify(gf, m, kv, cfg, prompt, k, rounds, seed, dev):
    """Verification passes of k drafts (gf_verify_k, k + 1 rows per pass) after
    the prompt: `rounds` passes whose drafts are the model's own greedy
    continuation (each pass accepts all k when no near-tie flips a token),
    then `rounds` passes with uniform random drafts (about none accepted).
    Returns the time per pass and the tokens each pass yields (accepted + 1)."""
    import numpy as np
    import torch
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
    seq = [int(t) for t in prompt]
    for t in prompt:
        tok.fill_(int(t))
        gf.decode_step(m, kv, tok, pos, logits, tok)
    seq.append(int(tok.item()))
    while len(seq) < N_PROMPT + rounds * (k + 1) + 1:
        gf.decode_step(m, kv, tok, pos, logits, tok)
        seq.append(int(tok.item()))
    starts = [N_PROMPT + r * (k + 1) for r in range(rounds)]
    rng = np.random.default_rng(seed)

    def passes(rows):
        pos_r = [torch.tensor([p], dtype=torch.int32, device=dev) for p in starts]
        tok_r = [torch.tensor(r_, dtype=torch.int32, device=dev) for r_ in rows]
        n_r = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in starts]
        x_r = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in starts]
        warm = torch.tensor([starts[0]], dtype=torch.int32, device=dev)
        gf.verify_k(m, kv, tok_r[0], k, warm, n_r[0], x_r[0])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record()
        for r in range(rounds):
            gf.verify_k(m, kv, tok_r[r], k, pos_r[r], n_r[r], x_r[r])
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1) / rounds
        acc = float(np.mean([int(n.item()) for n in n_r]))
        return {"ms_per_pass": round(ms, 4), "accepted_per_pass": acc, "tok_s": round((acc + 1) / (ms * 1e-3), 2)}

    greedy = passes([seq[p:p + k + 1] for p in starts])
    rand = passes([[seq[p]] + [int(x) for x in rng.integers(0, cfg["vocab"], k)] for p in starts])
    return {"k": k, "passes": rounds, "greedy_drafts": greedy, "random_drafts": rand,
            "device_error": gf.device_error()}


def measure_speculative(gf, cfg, glob, layers, prompt, args):
    """Speculative generation (gf_generate_speculative: draft = the
    --spec-draft copy of the same model proposing k tokens per round, target
    = the --spec-target copy verifying them) against plain greedy generation
    on the target (gf_generate), --spec-tokens tokens after the 5-token
    prompt, each call timed end to end on the host (the calls synchronise
    once per round / at the end) after one untimed call."""
    import torch
    k, n = args.speculate, args.spec_tokens
    tm = gf.Model(cfg, args.spec_target, glob, layers)
    dm = gf.Model(cfg, args.spec_draft, glob, layers)
    tmax = N_PROMPT + n + k + 8
    tkv, dkv = gf.KV(tm, tmax), gf.KV(dm, tmax)
    p = [int(t) for t in prompt]

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        r = fn()
        return r, time.perf_counter() - t0

    plain, t_plain = timed(lambda: gf.generate(tm, tkv, p, n))
    (toks, st), t_spec = timed(lambda: gf.generate_speculative(tm, tkv, dm, dkv, p, n, k))
    err = gf.device_error()
    for h in (tkv, dkv, tm, dm):
        h.close()
    # both calls include the prompt's N_PROMPT decode steps (and the draft's)
    return {"k": k, "target": args.spec_target, "draft": args.spec_draft, "tokens": n,
            "tok_s": round(n / t_spec, 2), "greedy_tok_s": round(n / t_plain, 2),
            "speedup": round(t_plain / t_spec, 3),
            "acceptance": round(st["accepted"] / max(st["drafted"], 1), 4), "rounds": st["rounds"],
            "same_tokens_as_greedy": toks == plain, "device_error": err,
            "timing": "host wall clock around each whole call (prompt included), after one untimed call"}


def measure_prefill(gf, cfg, glob, layers, prompt, args, dev):
    """The 5-token prompt as one gf_prefill pass (one weight stream for all
    rows) against 5 gf_decode_step calls, on the headline weights; CUDA
    events on the launching stream, median of 10 after 3 untimed."""
    import statistics as st
    import torch
    m = gf.Model(cfg, args.dtype, glob, layers)
    kv = gf.KV(m, 64)
    toks = torch.tensor([int(t) for t in prompt], dtype=torch.int32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    nxt = torch.zeros(1, dtype=torch.int32, device=dev)
    lg = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)

    def run_prefill():
        pos.zero_()
        gf.prefill(m, kv, toks, pos, nxt)

    def run_steps():
        pos.zero_()
        for i in range(len(prompt)):
            gf.decode_step(m, kv, toks[i:i + 1], pos, lg, nxt)

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(10):
            e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return st.median(ts)

    t_pre, t_steps = timed(run_prefill), timed(run_steps)
    err = gf.device_error()
    kv.close()
    m.close()
    return {"tokens": len(prompt), "weights": args.dtype, "prefill_ms": round(t_pre, 3),
            "decode_steps_ms": round(t_steps, 3), "device_error": err}


# ------------------------------------------------------------ our arm -----
def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from synth import models
    import weight_only_quantized_bs_gb300 as gf
    from weight_only_quantized_bs_gb300.weights import device_globals, fuse_layer

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    gf.lib()
    cfg = models.config(args.workload, group=args.group)
    if args.layers:
        cfg["n_layers"] = args.layers
    tmax, p_first, ctxs = bench_positions(args)
    dtypes = [args.dtype] if args.only_headline else ["int4", "int8", "bf16"]
    if args.dtype not in dtypes:
        dtypes.insert(0, args.dtype)

    # synthetic weights: drawn once on the host, fused, resident in HBM as bf16
    t0 = time.time()
    wc = models.WeightCache(cfg, seed=args.seed, keep=False)
    glob = device_globals(wc.glob, dev)
    layers = [fuse_layer(wc.layer(l), dev) for l in range(cfg["n_layers"])]
    torch.cuda.synchronize()
    gen_s = time.time() - t0
    prompt = models.prompt(cfg, args.seed, N_PROMPT)

    # copy ceiling of this GPU in this process: 1 GiB -> 1 GiB, 16-byte vectors
    nb = 1 << 30
    a = torch.empty(nb, dtype=torch.uint8, device=dev)
    b = torch.empty(nb, dtype=torch.uint8, device=dev)
    a.fill_(1)
    for _ in range(3):
        gf.copy_ceiling(a, b, nb)
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    best = 0.0
    for _ in range(10):
        e0.record()
        gf.copy_ceiling(a, b, nb)
        e1.record()
        e1.synchronize()
        best = max(best, 2 * nb / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    copy_gbs = best
    del a, b

    hbm_peak, peak_kind = measured_peaks()
    sampler = ClockSampler(local)
    results = {}
    stream = torch.cuda.current_stream()
    clocks = None
    for dt in dtypes:
        m = gf.Model(cfg, dt, glob, layers)
        kv = gf.KV(m, tmax)
        wbytes = m.weight_bytes()
        tok = torch.zeros(1, dtype=torch.int32, device=dev)
        pos = torch.zeros(1, dtype=torch.int32, device=dev)
        logits = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
        per_ctx = {}
        for ci, ctx in enumerate(ctxs or [None]):
            if ctx is None:
                # warm-up: the prompt, one token per step, then greedy steps
                for i in range(max(args.warmup, N_PROMPT)):
                    if i < N_PROMPT:
                        tok.fill_(int(prompt[i]))
                    gf.decode_step(m, kv, tok, pos, logits, tok)   # argmax -> next token
            else:
                # a context of ctx positions written into the cache, then greedy steps
                fill_context(gf, kv, cfg, args.seed, ctx, tmax, dev)
                pos.fill_(ctx)
                tok.fill_(int(prompt[0]))
                for i in range(args.warmup):
                    gf.decode_step(m, kv, tok, pos, logits, tok)
            torch.cuda.synchronize()
            p0 = int(pos.item())
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            head = dt == args.dtype and ci == 0
            if head:
                sampler.start()
                time.sleep(0.3)
            ev0, ev1 = torch.cuda.Event(True), torch.cuda.Event(True)
            ev0.record(stream)
            for _ in range(args.steps):
                gf.decode_step(m, kv, tok, pos, logits, tok)
            ev1.record(stream)
            ev1.synchronize()
            ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
            # repeat the timed loop for the clock record (not used for the number)
            if head:
                for _ in range(max(1, int(1500 / max(ms, 1)))):
                    for _ in range(args.steps):
                        gf.decode_step(m, kv, tok, pos, logits, tok)
                    torch.cuda.synchronize()
                    pos.fill_(p0)
                clocks = sampler.stop()
            err = gf.device_error()
            # algorithmic bytes: weights + KV rows 0..pos read + one row written, per token
            alg_bytes = decode_bytes(cfg, wbytes, p0, args.steps)
            toks = args.steps / (ms * 1e-3)
            gbs = alg_bytes / (ms * 1e-3) / 1e9
            rec = {"tok_s": toks * world, "ms_per_token": ms / args.steps, "gbs": gbs,
                   "frac_of_peak": gbs / hbm_peak, "frac_of_copy": gbs / copy_gbs,
                   "bytes_per_token": alg_bytes / args.steps, "weight_bytes": wbytes, "device_error": err}
            if ctx is not None:
                rec["ctx"] = ctx
            if ci == 0:
                # end to end through the C-ABI: token in from pinned host memory,
                # argmax out to pinned host memory, every step
                pos.fill_(p0)
                h_tok = torch.zeros(1, dtype=torch.int32).pin_memory()
                h_out = torch.zeros(1, dtype=torch.int32).pin_memory()
                h_tok[0] = int(prompt[-1])
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                for _ in range(args.steps):
                    tok.copy_(h_tok, non_blocking=True)
                    gf.decode_step(m, kv, tok, pos, logits, tok)
                    h_out.copy_(tok, non_blocking=True)
                    stream.synchronize()
                    h_tok[0] = h_out[0]
                e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
                rec["e2e_tok_s"] = args.steps / e2e_s * world
            per_ctx[ctx] = rec
        res = dict(per_ctx[(ctxs or [None])[0]])
        if ctxs:
            res["per_ctx"] = {str(c): per_ctx[c] for c in ctxs}
        if args.verify_k:
            res["verify"] = measure_verify(gf, m, kv, cfg, prompt, args.verify_k, 20, args.seed, dev)
        results[dt] = res
        kv.close()
        m.close()
        torch.cuda.synchronize()

    spec = measure_speculative(gf, cfg, glob, layers, prompt, args) if args.speculate else None
    pre = measure_prefill(gf, cfg, glob, layers, prompt, args, dev) if args.prefill else None
    head = results[args.dtype]
    out = {
        "metric": METRIC,
        "value": round(head["tok_s"], 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, N_PROMPT),
        "ms_per_step": round(head["ms_per_token"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "vs_published_a100": ({"ratio": round(head["tok_s"] / world / PUBLISHED_TOKS[(args.workload, args.dtype)], 3),
                               "published_tok_s": PUBLISHED_TOKS[(args.workload, args.dtype)],
                               "hardware": "1x A100-80GB at 330 W (gpt-fast README, Benchmarks); context only"}
                              if (args.workload, args.dtype) in PUBLISHED_TOKS else None),
        "dtype": "f32",
        "data": "synthetic (seeded random-init weights, uniform random prompt)",
        "config": bench_config(args, cfg, tmax, p_first, ctxs),
        "achieved_gbs": round(head["gbs"], 1),
        "roofline": {"bound": "hbm", "achieved": round(head["gbs"], 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(head["gbs"] / hbm_peak, 4),
                     "traffic": measured_traffic(args.workload, args.dtype),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (%s)" % peak_kind,
                     "kernel": "k_engine (one launch per token)"},
        "copy_ceiling_gbs": round(copy_gbs, 1),
        "per_dtype": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                      for k, v in results.items()},
        "e2e": {"value": round(head["e2e_tok_s"], 2), "unit": "tokens/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "setup_s": round(gen_s, 1),
    }
    if spec is not None:
        out["speculative"] = spec
    if pre is not None:
        out["prefill"] = pre
    del layers, glob
    if rank == 0 and not args.no_cpu_baseline:
        # the token stream from the first timed position, stage by stage, for
        # about 20 s of CPU (at most one whole token); only the layers the
        # sample reaches are built
        probe = OracleStream(cfg, args.dtype, args.seed, p_first, 1)
        t1 = probe.stage()
        n = max(1, min(cfg["n_layers"] + 1, int(20.0 / max(t1, 1e-3))))
        del probe
        st = OracleStream(cfg, args.dtype, args.seed, p_first, n)
        spent = sum(st.stage() for _ in range(n))
        out["cpu_baseline"] = {"value": round(n / st.n_stages / spent, 5), "unit": "tokens/s", "cores": 1,
                               "kind": "oracle",
                               "sample": "%d stages (of %d per token: %d layers + lm_head) of the token stream at "
                                         "position %d, %.1f s on one core; value = stages / %d per second "
                                         "(building and quantising the layers untimed)"
                                         % (n, st.n_stages, cfg["n_layers"], p_first, spent, st.n_stages)}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------- GEMV workloads ---
GEMV_SET = [("qkv", 12288, 4096), ("o", 4096, 4096), ("gate_up", 22016, 4096), ("down", 4096, 11008),
            ("lm_head", 32000, 4096)]


def run_gemv(args):
    """Standalone GEMVs: the Llama-2-7B layer set (gemv-set) or the single
    4096 x 4096 GEMV (gemv), x ~ N(0,1), W ~ N(0,0.02).  Distinct weight copies
    totalling at least 4x L2 rotate through the timed loop."""
    import torch
    import __graft_entry__
    import synth
    import weight_only_quantized_bs_gb300 as gf
    from weight_only_quantized_bs_gb300.weights import to_dev
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes = GEMV_SET if args.workload == "gemv-set" else [("single", 4096, 4096)]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    dt = gf.DTYPE_NAMES[args.dtype]
    per = []
    for name, N, K in shapes:
        W = to_dev(synth.normal_bf16(args.seed, 700 + N % 97, (N, K), 0.02))
        if dt == gf.W_INT8:
            qp, s8 = gf.quantize_w8(W)
        elif dt == gf.W_INT4G32:
            qp, s8 = gf.quantize_w4g(W), None
        else:
            qp, s8 = gf.repack_bf16(W), None
        del W
        nbytes = qp.numel() + (s8.numel() * 2 if s8 is not None else 0) + 2 * K + 4 * N
        copies = max(1, -(-4 * l2 // nbytes))
        packs = [qp] + [qp.clone() for _ in range(copies - 1)]
        x = to_dev(synth.normal_bf16(args.seed, 5, (K,), 1.0))
        y = torch.empty(N, dtype=torch.float32, device=dev)

        def call(i):
            p = packs[i % copies]
            if dt == gf.W_INT8:
                gf.gemv_w8(x, p, s8, N, K, gf.Y_F32, out=y)
            elif dt == gf.W_INT4G32:
                gf.gemv_w4g(x, p, N, K, gf.Y_F32, out=y)
            else:
                gf.gemv_bf16(x, p, N, K, gf.Y_F32, out=y)
        for i in range(args.warmup):
            call(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record()
        for i in range(args.steps):
            call(i)
        e1.record()
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        per.append({"name": name, "N": N, "K": K, "bytes": nbytes, "us": round(us, 2),
                    "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "copies": copies})
        del packs
    tot_b = sum(p["bytes"] for p in per)
    tot_us = sum(p["us"] for p in per)
    hbm_peak, kind = measured_peaks()
    gbs = tot_b / (tot_us * 1e-6) / 1e9
    print(json.dumps({
        "metric": "standalone GEMV GB/s (%s)" % args.workload, "value": round(gbs, 1), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_us / 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": args.workload, "weights": args.dtype,
                                        "l2": "weights rotate through copies totalling >= 4x L2"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(gbs / hbm_peak, 4), "traffic": None},
        "per_gemv": per, "gpu_launches": args.steps * len(shapes)}))


# ------------------------------------------------------ reference arm -----
def run_reference(args):
    """The oracle (this build's reference implementation) on the host: the
    same command's workload as a stream of token stages (OracleStream), one
    stage per step after `warmup` untimed stages.  value = the stages timed /
    (n_layers + 1) per second: whole-token throughput measured on the stages
    run (every stage of a token is one layer or the lm_head; a run of fewer
    than n_layers + 1 steps measures part of a token's work)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from synth import models
    cfg = models.config(args.workload, group=args.group)
    if args.layers:
        cfg["n_layers"] = args.layers
    tmax, p_first, ctxs = bench_positions(args)
    st = OracleStream(cfg, args.dtype, args.seed, p_first, args.warmup + args.steps)
    for _ in range(args.warmup):
        st.stage()
    t0 = time.perf_counter()
    per = [st.stage() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    v = args.steps / st.n_stages / wall
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded random-init weights, uniform random prompt)",
        "config": bench_config(args, cfg, tmax, p_first, ctxs),
        "cpu_baseline": {"value": round(v, 5), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "%d stages (of %d per token: %d layers + lm_head) of the token stream "
                                   "from position %d after %d untimed stages; stage times %.3f-%.3f s"
                                   % (args.steps, st.n_stages, cfg["n_layers"], p_first, args.warmup,
                                      min(per), max(per))},
        "e2e": {"value": round(v, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.workload in ("gemv-set", "gemv"):
        run_gemv(a)
    else:
        run_ours(a)
