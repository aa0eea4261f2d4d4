#!/usr/bin/env python
"""Benchmark of one EAGLE-2 tree-verify step on GB300: draft-tree build,
tree-masked GQA attention, acceptance walk (all three through the C ABI).

Default workload: Qwen2-7B layer shape at 8K context (28 q / 4 kv heads,
d 128, bf16 KV prefix 8192; vocab 152064; top_k 10, depth 6, 60-token tree;
sampling T 0.7, top_k 50, top_p 0.9), synthetic seeded inputs.

Prints ONE JSON line (rank 0).  `value` = microseconds per verify step with
every input resident in HBM, L2 flushed before each step (inputs 86 MB < L2),
step replayed as a CUDA graph; `e2e` = the same step with the per-step inputs
copied from pinned host memory and the accepted path read back.
--impl reference times the fp64 CPU oracle on the same workload (host cores).
With torchrun (N > 1) every rank runs an independent replica (weak scaling).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per tree-verify step and tree-attn HBM GB/s (% of peak) at 8K ctx"
NAMES = ("q", "k_cache", "v_cache", "tree_k", "tree_v")
WORKLOAD_LABEL = {
    "c0": "tiny: vocab 1000, 16-token tree, 4/2 heads d64 fp32, prefix 128, greedy",
    "c1": "llama3-8b layer: vocab 128256, 60-token tree, 32/8 heads d128, prefix 2048, greedy",
    "c2": "qwen2-7b layer: vocab 152064, 60-token tree (top_k 10, depth 6), 28/4 heads d128, "
          "bf16 prefix 8192, sampling T0.7 top_k50 top_p0.9",
    "c3": "llama3-8b, 32 layers x prefix 32768: vocab 128256, 60-token tree, greedy",
    "c4": "16 ragged sequences, prefixes U[512,16384], 64/8 heads d128, vocab 128256",
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = self.rows
        if self.window:
            t0, t1 = self.window
            inside = [r for r in rows if t0 - 0.06 <= r[0] <= t1 + 0.06]
            rows = inside or rows
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, v in rows:
            try:
                sm.append(float(v[0]))
                smax = max(smax, float(v[1]))
                for n, flag in zip(names, v[4:8]):
                    if flag.lower().startswith("active"):
                        reasons.add(n)
            except Exception:
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm
# the sources each timed kernel is compiled from (its .cu and every header
# it includes, directly or not)
KERNEL_SOURCES = {
    "build": ["eagle_build.cu", "eagle_stream_host.h", "eagle_rowstream.cuh", "eagle_host.h",
              "eagle_common.cuh"],
    "verify": ["eagle_verify.cu", "eagle_philox.cuh", "eagle_stream_host.h", "eagle_rowstream.cuh",
               "eagle_host.h", "eagle_common.cuh"],
    "attn": ["eagle_attn_tc.cu", "eagle_attn.cu", "eagle_attn.h", "eagle_tc.cuh", "eagle_host.h",
             "eagle_common.cuh"],
}


def _kernel_source_hash(kernel):
    """sha1 of one kernel's sources with comments and blank lines removed, so
    that editing a comment, or another kernel, does not void its recorded
    traffic figures."""
    import re
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "eagle_speculative_decoding_verify_gb300", "csrc")
    used = set()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.normpath(os.path.join(csrc, name)), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        used |= set(re.findall(r"\bEAGLE_[A-Z0-9_]+\b", text))
        h.update(os.path.basename(name).encode())
        h.update("\n".join(lines).encode())
    # of the public header, the constants these sources use (limits, status codes)
    with open(os.path.join(ROOT, "include", "eagle.h"), encoding="utf-8") as f:
        consts = []
        for ln in f:
            mt = re.match(r"\s*(?:#define\s+)?(EAGLE_[A-Z0-9_]+)(?:\s+|\s*=)", ln)
            if mt and mt.group(1) in used and ("#define" in ln or "=" in ln):
                consts.append(ln.split("/*")[0].strip())
    h.update("\n".join(sorted(consts)).encode())
    return h.hexdigest()[:12]


class Step:
    """Device buffers and the three calls of one verify step (single sequence)."""

    def __init__(self, w, dev, eb, wl):
        import torch
        self.torch, self.eb, self.w = torch, eb, w
        self.draft_h = wl.draft_logits(w)
        self.root = wl.root_token(w)
        a = wl.attention_inputs(w)
        self.attn_h = {n: a[n] for n in NAMES}
        self.draft = self.draft_h.to(dev)
        self.attn = {n: t.to(dev) for n, t in self.attn_h.items()}
        self.tree = eb.Tree(w.total_tokens, dev)
        self.ws_build = eb.workspace(eb.eagle_tree_build_workspace_size(
            1, w.n_rows, w.vocab, w.top_k, w.depth, w.total_tokens), dev)
        dtype = eb.EAGLE_BF16 if w.dtype == "bf16" else eb.EAGLE_F32
        self.out = torch.empty(w.total_tokens, w.n_q_heads, w.head_dim, device=dev)
        self.ws_attn = eb.workspace(eb.eagle_tree_attn_workspace_size(
            w.total_tokens, w.n_q_heads, w.n_kv_heads, w.head_dim, w.prefix, dtype), dev)
        self.item = eb.attn_item(self.attn["q"], self.attn["k_cache"], self.attn["v_cache"],
                                 self.attn["tree_k"], self.attn["tree_v"], self.tree.mask,
                                 self.out)
        self.attn_launches = eb.eagle_tree_attn_num_launches(
            [self.item], w.n_q_heads, w.n_kv_heads, w.head_dim, dtype)
        gr, T, k, p = w.sampling_of(0)
        self.params = eb.sampling(gr, T, k, p)
        # target logits depend on the tree: build it once (untimed) on the GPU
        eb.eagle_tree_build(self.draft, w.top_k, w.depth, w.total_tokens, self.root,
                            out=self.tree, ws=self.ws_build)
        torch.cuda.synchronize()
        self.target_h = wl.target_logits(w, self.tree.parents.cpu().tolist(),
                                         self.tree.tokens.cpu().tolist())
        self.target = self.target_h.to(dev)
        self.ws_verify = eb.workspace(eb.eagle_tree_verify_workspace_size(
            1, w.total_tokens, w.vocab), dev)
        self.acc = torch.zeros(w.total_tokens, dtype=torch.int32, device=dev)
        self.n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
        self.bonus = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches = 1 + self.attn_launches + 1

    def build(self, s):
        w = self.w
        self.eb.eagle_tree_build(self.draft, w.top_k, w.depth, w.total_tokens, self.root,
                                 out=self.tree, ws=self.ws_build, stream=s)

    def attention(self, s):
        w = self.w
        a = self.attn
        self.eb.eagle_tree_attn(a["q"], a["k_cache"], a["v_cache"], a["tree_k"], a["tree_v"],
                                self.tree.mask, out=self.out, ws=self.ws_attn, stream=s)

    def verify(self, s, step=0):
        self.eb.eagle_tree_verify(self.target, self.tree, self.params, 1234, step,
                                  accepted=self.acc, n_accepted=self.n_acc,
                                  bonus_token=self.bonus, ws=self.ws_verify, stream=s)

    def run(self, s):
        self.build(s)
        self.attention(s)
        self.verify(s)

    # algorithmic bytes / flops
    def bytes_build(self):
        w = self.w
        return w.n_rows * w.vocab * 4

    def bytes_verify(self):
        w = self.w
        return w.total_tokens * w.vocab * 4

    def bytes_attn(self):
        w = self.w
        el = 2 if w.dtype == "bf16" else 4
        kv = 2 * w.prefix * w.n_kv_heads * w.head_dim * el
        q = w.total_tokens * w.n_q_heads * w.head_dim * el
        tkv = 2 * w.total_tokens * w.n_kv_heads * w.head_dim * el
        out = w.total_tokens * w.n_q_heads * w.head_dim * 4
        return kv + q + tkv + out

    def flops_attn(self):
        w = self.w
        return 4.0 * w.total_tokens * w.n_q_heads * (w.prefix + w.total_tokens) * w.head_dim

    def h2d_bytes(self):
        return (self.draft_h.numel() * 4 + self.target_h.numel() * 4 +
                sum(self.attn_h[n].numel() * self.attn_h[n].element_size()
                    for n in ("q", "tree_k", "tree_v")))


class MultiStep:
    """One verify step of any workload through the batched entry points: the
    items' trees in one build launch, every attention problem (a layer of the
    long-context workload, or a sequence of the ragged batch) in one batched
    attention call, every item's walk in one verify launch."""

    def __init__(self, w, dev, eb, wl):
        import torch
        self.torch, self.eb, self.w = torch, eb, w
        n, m = w.items, w.total_tokens
        self.draft = [wl.draft_logits(w, b).to(dev) for b in range(n)]
        self.roots = [wl.root_token(w, b) for b in range(n)]
        self.trees = [eb.Tree(m, dev) for _ in range(n)]
        self.ws_build = eb.workspace(eb.eagle_tree_build_workspace_size(
            n, w.n_rows, w.vocab, w.top_k, w.depth, m), dev)
        self.build(torch.cuda.current_stream())          # untimed: the target logits need the trees
        torch.cuda.synchronize()
        self.target = [wl.target_logits(w, t.parents.cpu().tolist(), t.tokens.cpu().tolist(),
                                        b).to(dev) for b, t in enumerate(self.trees)]
        self.prefix = wl.prefix_lengths(w)
        self.dtype = eb.EAGLE_BF16 if w.dtype == "bf16" else eb.EAGLE_F32
        self.attn, self.outs, self.items = [], [], []
        problems = ([(0, l) for l in range(w.layers)] if w.layers > 1 else
                    [(b, 0) for b in range(n)])
        for b, l in problems:
            a = wl.attention_inputs(w, item=b, layer=l, device=dev, prefix=self.prefix[b])
            o = torch.empty(m, w.n_q_heads, w.head_dim, device=dev)
            self.attn.append(a)
            self.outs.append(o)
            self.items.append(eb.attn_item(a["q"], a["k_cache"], a["v_cache"], a["tree_k"],
                                           a["tree_v"], self.trees[b].mask, o))
        self.ws_attn = eb.workspace(eb.eagle_tree_attn_batched_workspace_size(
            self.items, w.n_q_heads, w.n_kv_heads, w.head_dim, self.dtype), dev)
        self.attn_launches = eb.eagle_tree_attn_num_launches(
            self.items, w.n_q_heads, w.n_kv_heads, w.head_dim, self.dtype)
        self.params = [eb.sampling(*w.sampling_of(b)) for b in range(n)]
        self.seeds = [1234 + b for b in range(n)]
        self.ws_verify = eb.workspace(eb.eagle_tree_verify_workspace_size(n, m, w.vocab), dev)
        self.acc = [torch.zeros(m, dtype=torch.int32, device=dev) for _ in range(n)]
        self.n_acc = torch.zeros(n, dtype=torch.int32, device=dev)
        self.bonus = torch.zeros(n, dtype=torch.int32, device=dev)
        self.launches = 1 + self.attn_launches + 1

    def build(self, s):
        w = self.w
        self.eb.eagle_tree_build_batched(self.draft, w.top_k, w.depth, w.total_tokens, self.roots,
                                         outs=self.trees, ws=self.ws_build, stream=s)

    def attention(self, s):
        w = self.w
        self.eb.eagle_tree_attn_batched(self.items, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                        self.dtype, ws=self.ws_attn, stream=s)

    def verify(self, s, step=0):
        self.eb.eagle_tree_verify_batched(self.target, self.trees, self.params, self.seeds, step,
                                          accepted=self.acc, n_accepted=self.n_acc,
                                          bonus_tokens=self.bonus, ws=self.ws_verify, stream=s)

    def run(self, s):
        self.build(s)
        self.attention(s)
        self.verify(s)

    def bytes_build(self):
        w = self.w
        return w.items * w.n_rows * w.vocab * 4

    def bytes_verify(self):
        w = self.w
        return w.items * w.total_tokens * w.vocab * 4

    def _problems(self):
        w = self.w
        return [(self.prefix[0], ) for _ in range(w.layers)] if w.layers > 1 else \
            [(self.prefix[b], ) for b in range(w.items)]

    def bytes_attn(self):
        w = self.w
        el = 2 if w.dtype == "bf16" else 4
        m, hq, hkv, d = w.total_tokens, w.n_q_heads, w.n_kv_heads, w.head_dim
        return sum(2 * S * hkv * d * el + m * hq * d * el + 2 * m * hkv * d * el + m * hq * d * 4
                   for (S, ) in self._problems())

    def flops_attn(self):
        w = self.w
        m, hq, d = w.total_tokens, w.n_q_heads, w.head_dim
        return sum(4.0 * m * hq * (S + m) * d for (S, ) in self._problems())


def config_bench(eb, wl, dev, key, flush, K):
    """µs per verify step of one workload (CUDA graph, L2 flushed before every
    step), the per-call split, and the step's roofline fraction (HBM time of
    the logit passes plus the attention's larger of HBM and tensor time,
    against the measured peaks)."""
    import torch
    w = wl.WORKLOADS[key]
    st = MultiStep(w, dev, eb, wl)
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for _ in range(3):
            flush.zero_()
            st.run(s)
    s.synchronize()
    times, _ = _time_graph(torch, st, s, flush, K)
    per = _time_kernels(torch, st, s, flush, K)
    hbm, tf, _, peak_src = _peaks()
    k_us = {k: statistics.mean(v) for k, v in per.items()}
    roof_us = {"build": st.bytes_build() / (hbm * 1e3), "verify": st.bytes_verify() / (hbm * 1e3),
               "attn": max(st.bytes_attn() / (hbm * 1e3), st.flops_attn() / (tf * 1e6))}
    us = statistics.mean(times)
    err = [eb.workspace_error(ws, s)[0] for ws in (st.ws_build, st.ws_attn, st.ws_verify)]
    assert err == [0, 0, 0], f"{key}: device error words {err}"
    res = {"workload": WORKLOAD_LABEL[key], "us_per_step": round(us, 2),
           "spread_us": spread(times), "kernels_us": {k: round(v, 2) for k, v in k_us.items()},
           "roofline_us": {k: round(v, 3) for k, v in roof_us.items()},
           "step_roofline_us": round(sum(roof_us.values()), 3),
           "step_roofline_frac": round(sum(roof_us.values()) / us, 4),
           "attn_frac_hbm": round(st.bytes_attn() / (k_us["attn"] * 1e3) / hbm, 4),
           "attn_frac_tensor": round(st.flops_attn() / (k_us["attn"] * 1e6) / tf, 4),
           "bytes": {"build": st.bytes_build(), "attn": st.bytes_attn(),
                     "verify": st.bytes_verify()},
           "attn_gflop": round(st.flops_attn() / 1e9, 3), "launches": st.launches,
           "items": w.items, "layers": w.layers, "steps": K, "peak_source": peak_src}
    del st
    torch.cuda.empty_cache()
    return res


def oracle_one_thread(key):
    """The oracle's step on ONE host thread (BLAS pinned to one thread in a
    child process, since the setting must precede numpy's import)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    code = ("import json, bench; r = bench.cpu_baseline(%r, samples=1); r['cores'] = 1; "
            "print(json.dumps(r))" % key)
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                             text=True, timeout=600)
        line = [ln for ln in out.stdout.splitlines() if ln.startswith("{")][-1]
        return json.loads(line)
    except Exception as exc:
        return {"error": str(exc)[:200]}


def attn_long(eb, wl, dev, reps=5, n_layers=None, paged=True, fp8=True):
    """Tree attention at long context: 32 independent layers of a
    llama-3-8b-shaped KV cache (8 kv heads, d 128, bf16 prefix 32768; 4.3 GB,
    far above L2) for one 60-token tree, all layers in one batched call
    (n_layers of them when given: a smaller case of the same kernel, for
    profiling).  Returns achieved GB/s (algorithmic bytes / device time) and
    TFLOP/s."""
    import torch
    w = wl.WORKLOADS["c3"]
    nl = w.layers if n_layers is None else n_layers
    draft = wl.draft_logits(w).to(dev)
    tree = eb.eagle_tree_build(draft, w.top_k, w.depth, w.total_tokens, wl.root_token(w))
    layers = [wl.attention_inputs(w, layer=l, device=dev) for l in range(nl)]
    outs = [torch.empty(w.total_tokens, w.n_q_heads, w.head_dim, device=dev)
            for _ in range(nl)]
    items = [eb.attn_item(a["q"], a["k_cache"], a["v_cache"], a["tree_k"], a["tree_v"],
                          tree.mask, o) for a, o in zip(layers, outs)]
    dt = eb.EAGLE_BF16
    ws = eb.workspace(eb.eagle_tree_attn_batched_workspace_size(
        items, w.n_q_heads, w.n_kv_heads, w.head_dim, dt), dev)
    s = torch.cuda.Stream(device=dev)

    def run():
        eb.eagle_tree_attn_batched(items, w.n_q_heads, w.n_kv_heads, w.head_dim, dt, ws=ws,
                                   stream=s, device=dev)

    for _ in range(2):
        run()
    s.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        run()
        e1.record(s)
        s.synchronize()
        times.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(times)
    m, hq, hkv, d, S, L = w.total_tokens, w.n_q_heads, w.n_kv_heads, w.head_dim, w.prefix, nl
    nbytes = L * (2 * S * hkv * d * 2 + m * hq * d * 2 + 2 * m * hkv * d * 2 + m * hq * d * 4)
    flops = L * 4.0 * m * hq * (S + m) * d
    res = {"workload": f"c3: {nl} layers x bf16 prefix 32768, 32/8 heads d128, 60-token tree, "
                       "one batched call", "us": round(t * 1e6, 1),
           "achieved_gbs": round(nbytes / t / 1e9, 1),
           "achieved_tflops": round(flops / t / 1e12, 1), "bytes": nbytes}
    if paged:   # the same keys / values in 128-token pages, shuffled within each layer's pool
        page = eb.EAGLE_KV_PAGE_TOKENS
        n_pages = S // page
        gen = torch.Generator().manual_seed(5)
        pitems, keep = [], []
        for a, o in zip(layers, outs):
            perm = torch.randperm(n_pages, generator=gen)
            table = torch.argsort(perm).to(torch.int32).to(dev)   # page j at pool page table[j]
            kp = a["k_cache"].view(hkv, n_pages, page, d)[:, perm].reshape(hkv, S, d).contiguous()
            vp = a["v_cache"].view(hkv, n_pages, page, d)[:, perm].reshape(hkv, S, d).contiguous()
            keep.append((kp, vp, table))
            pitems.append(eb.attn_paged_item(a["q"], kp, vp, table, a["tree_k"], a["tree_v"],
                                             tree.mask, o, S))
        pws = eb.workspace(eb.lib().eagle_tree_attn_paged_workspace_size(
            (eb.CAttnPagedItem * nl)(*pitems), nl, hq, hkv, d), dev)

        def run_paged():
            eb.eagle_tree_attn_paged_batched(pitems, hq, hkv, d, ws=pws, stream=s)

        for _ in range(2):
            run_paged()
        s.synchronize()
        ptimes = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            run_paged()
            e1.record(s)
            s.synchronize()
            ptimes.append(e0.elapsed_time(e1) * 1e-3)
        pt = statistics.median(ptimes)
        res["paged"] = {"us": round(pt * 1e6, 1), "achieved_gbs": round(nbytes / pt / 1e9, 1),
                        "page_tokens": page, "pages_shuffled": True}
        del keep, pitems, pws
    if fp8:   # the same prefixes as E4M3 codes with one scale per (kv head, 128-token page)
        fitems, fkeep = [], []
        for a, o in zip(layers, outs):
            kc, ks = wl.fp8_kv(a["k_cache"])
            vc, vs = wl.fp8_kv(a["v_cache"])
            fkeep.append((kc, ks, vc, vs))
            fitems.append(eb.attn_fp8_item(a["q"], kc, vc, ks, vs, a["tree_k"], a["tree_v"],
                                           tree.mask, o, S))
        fws = eb.workspace(eb.lib().eagle_tree_attn_fp8_workspace_size(
            (eb.CAttnFp8Item * nl)(*fitems), nl, hq, hkv, d), dev)

        def run_fp8():
            eb.eagle_tree_attn_fp8_batched(fitems, hq, hkv, d, ws=fws, stream=s)

        for _ in range(2):
            run_fp8()
        s.synchronize()
        ftimes = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            run_fp8()
            e1.record(s)
            s.synchronize()
            ftimes.append(e0.elapsed_time(e1) * 1e-3)
        ft = statistics.median(ftimes)
        fbytes = L * (2 * S * hkv * d * 1 + 2 * hkv * (S // 128) * 4 + m * hq * d * 2 +
                      2 * m * hkv * d * 2 + m * hq * d * 4)
        res["fp8"] = {"us": round(ft * 1e6, 1), "achieved_gbs": round(fbytes / ft / 1e9, 1),
                      "bytes": fbytes, "achieved_tflops": round(flops / ft / 1e12, 1),
                      "format": "E4M3 codes, one fp32 scale per (kv head, 128-token page)"}
        del fkeep, fitems, fws
    del layers, outs, items, ws
    torch.cuda.empty_cache()
    return res


def kv_commit_bench(eb, wl, dev, step, s, reps=200):
    """The KV commit after acceptance (append the accepted path's keys and
    values to the prefix cache): device time of one call for the c2 layer and
    of one batched call over the 32 layers of the c3 shape (32K prefix each),
    for the path to a deepest node of the step's tree (root + one node per depth), each
    call replayed from a CUDA graph.  Tens of KB to 1 MB move per call, so
    the figure is a latency, reported with its bytes (read + written)."""
    import torch
    w = step.w
    parents = step.tree.parents.cpu().tolist()
    depth = step.tree.depth.cpu().tolist()
    node = max(range(len(depth)), key=lambda i: (depth[i], -i))   # a deepest node
    path = []
    while node >= 0:   # its ancestors, root first
        path.append(node)
        node = parents[node]
    path = path[::-1]
    acc = torch.zeros(w.total_tokens, dtype=torch.int32, device=dev)
    acc[: len(path)] = torch.tensor(path, dtype=torch.int32, device=dev)
    n_acc = torch.tensor([len(path) - 1], dtype=torch.int32, device=dev)
    rows = len(path)
    m, hkv, d = w.total_tokens, w.n_kv_heads, w.head_dim
    el = 2 if w.dtype == "bf16" else 4
    kc = torch.empty(hkv, w.prefix + m, d, dtype=step.attn["k_cache"].dtype, device=dev)
    vc = torch.empty_like(kc)
    ws = eb.workspace(eb.eagle_kv_commit_workspace_size(), dev)

    def timed(fn):
        for _ in range(3):
            fn()
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            graph.replay()
        e1.record(s)
        s.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    c2_us = timed(lambda: eb.eagle_kv_commit(kc, vc, step.attn["tree_k"], step.attn["tree_v"],
                                             acc, n_acc, w.prefix, ws=ws, stream=s))
    w3 = wl.WORKLOADS["c3"]
    L3, S3 = w3.layers, w3.prefix
    g = torch.Generator(device=dev).manual_seed(7)
    items, keep = [], []
    for _ in range(L3):
        k3 = torch.empty(w3.n_kv_heads, S3 + m, w3.head_dim, dtype=torch.bfloat16, device=dev)
        v3 = torch.empty_like(k3)
        tk = torch.randn(m, w3.n_kv_heads, w3.head_dim, generator=g, device=dev).to(torch.bfloat16)
        tv = torch.randn(m, w3.n_kv_heads, w3.head_dim, generator=g, device=dev).to(torch.bfloat16)
        keep.append((k3, v3, tk, tv))
        items.append(eb.kv_item(k3, v3, tk, tv, acc, n_acc, S3))
    c3_us = timed(lambda: eb.eagle_kv_commit_batched(items, w3.n_kv_heads, w3.head_dim,
                                                     eb.EAGLE_BF16, ws=ws, stream=s))
    st, _ = eb.workspace_error(ws, s)
    assert st == 0, f"kv commit device error {st}"
    b2 = 2 * 2 * rows * hkv * d * el
    b3 = L3 * 2 * 2 * rows * w3.n_kv_heads * w3.head_dim * 2
    del keep, items
    return {"rows": rows, "c2_us": round(c2_us, 2), "c2_bytes": b2,
            "c3_32layers_us": round(c3_us, 2), "c3_bytes": b3,
            "c3_achieved_gbs": round(b3 / (c3_us * 1e-6) / 1e9, 1)}


def tree_expand_bench(eb, wl, dev, step, s, flush, reps=50):
    """The per-depth tree build of a drafting round (one eagle_tree_expand
    call per depth on that depth's draft rows, then eagle_tree_finalize) on
    the step's draft logits, replayed from a CUDA graph with L2 flushed before
    every round; the tree must equal the one-shot build's."""
    import torch
    w = step.w
    k, D, m, V = w.top_k, w.depth, w.total_tokens, w.vocab
    g = eb.TreeGrowth(k, D, V, dev)
    out = eb.Tree(m, dev)
    rows = [step.draft[0:1]] + [step.draft[1 + (l - 1) * k: 1 + l * k] for l in range(1, D)]

    def round_():
        for level in range(D):
            g.expand(rows[level], level, stream=s)
        g.finalize(m, step.root, out=out, stream=s)

    for _ in range(3):
        round_()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        round_()
    times = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        graph.replay()
        e1.record(s)
        s.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    st, _ = eb.workspace_error(g.ws, s)
    same = (st == 0 and torch.equal(out.parents, step.tree.parents) and
            torch.equal(out.mask, step.tree.mask))
    assert same, "per-depth build differs from the one-shot build"
    return {"us_per_round": round(statistics.median(times), 2), "launches": D + 1,
            "bytes": (1 + (D - 1) * k) * V * 4,
            "note": "L2 flushed before each round; rows of every depth from HBM"}


def verify_nucleus_bench(eb, wl, dev, step, s, flush, reps=50):
    """The step's verify with the nucleus over the whole vocabulary (T 0.7,
    top_p 0.9, no top_k) instead of top_k 50: one call, replayed from a CUDA
    graph with L2 flushed before every call, beside the same call with the
    workload's own sampling."""
    import torch
    out = {}
    for name, params in (("nucleus", eb.sampling(False, 0.7, 0, 0.9)), ("workload", step.params)):
        def call():
            eb.eagle_tree_verify(step.target, step.tree, params, 1234, 0, accepted=step.acc,
                                 n_accepted=step.n_acc, bonus_token=step.bonus, ws=step.ws_verify,
                                 stream=s)

        for _ in range(3):
            call()
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            call()
        times = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            graph.replay()
            e1.record(s)
            s.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        assert eb.workspace_error(step.ws_verify, s)[0] == 0, "verify recorded a device error"
        out[name + "_us"] = round(statistics.median(times), 2)
    out["sampling"] = "nucleus: T 0.7, top_k 0, top_p 0.9; workload: T 0.7, top_k 50, top_p 0.9"
    out["note"] = "L2 flushed before each call; one launch per call"
    return out


def tree_policy_bench(eb, wl, dev, step, s, flush, reps=50):
    """The tree-shape policies on the step's draft logits (51 rows of the
    vocabulary): the confidence-ratio tree (tau 2, up to 4 branches, depth <= 7,
    at most 52 nodes: one row per possible inner node) and 10 batched chains
    of depth 6 (61 nodes, the 51 rows exactly); one call each, replayed from a
    CUDA graph with L2 flushed before every call."""
    import torch
    V = step.w.vocab
    n_rows = step.draft.shape[0]
    cases = {"confidence": (eb.tree_policy(eb.EAGLE_POLICY_CONFIDENCE, 4, 7, 2.0), n_rows + 1),
             "chains_10x6": (eb.tree_policy(eb.EAGLE_POLICY_CHAINS, 10, 6), 61)}
    res = {}
    for name, (pol, m) in cases.items():
        ws = eb.workspace(eb.eagle_tree_policy_workspace_size(V, pol, m), dev)
        out = eb.Tree(m, dev, with_values=False)
        nn = torch.zeros(1, dtype=torch.int32, device=dev)

        def call():
            eb.eagle_tree_build_policy(step.draft, pol, m, step.root, out=out, n_nodes=nn, ws=ws,
                                       stream=s)

        for _ in range(3):
            call()
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            call()
        times = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            graph.replay()
            e1.record(s)
            s.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        assert eb.workspace_error(ws, s)[0] == 0, "policy build recorded a device error"
        rows = min(n_rows, m - 1)
        us = statistics.median(times)
        res[name] = {"us": round(us, 2), "nodes": int(nn.item()), "rows": rows,
                     "bytes": rows * V * 4, "achieved_gbs": round(rows * V * 4 / us / 1e3, 1)}
    res["note"] = "L2 flushed before each call; one launch per call"
    return res


class L2Flush:
    """Evicts the step's inputs from L2 before every step: writes 512 MB (4x
    L2), then reads 256 MB so that the lines left behind are clean and the
    timed step does not pay for writing back the flush's dirty lines."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.sink = torch.zeros(1, dtype=torch.float32, device=dev)

    def zero_(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


def _time_graph(torch, step, s, flush, K):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step.run(s)          # warm the allocator-free path once outside capture
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        step.run(s)
    times = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    with torch.cuda.stream(s):
        for e0, e1 in ev:
            flush.zero_()
            e0.record(s)
            g.replay()
            e1.record(s)
    s.synchronize()
    for e0, e1 in ev:
        times.append(e0.elapsed_time(e1) * 1e3)
    return times, g


def _time_kernels(torch, step, s, flush, K):
    """Per-call device times (µs) with events between the calls."""
    per = {"build": [], "attn": [], "verify": []}
    evs = []
    with torch.cuda.stream(s):
        for _ in range(K):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            flush.zero_()
            e[0].record(s)
            step.build(s)
            e[1].record(s)
            step.attention(s)
            e[2].record(s)
            step.verify(s)
            e[3].record(s)
            evs.append(e)
    s.synchronize()
    for e in evs:
        per["build"].append(e[0].elapsed_time(e[1]) * 1e3)
        per["attn"].append(e[1].elapsed_time(e[2]) * 1e3)
        per["verify"].append(e[2].elapsed_time(e[3]) * 1e3)
    return per


def _time_e2e(torch, step, s, flush, K):
    """Same step with per-step inputs from pinned host memory and the result
    read back; device-timed around copies + calls.  The target logits, which
    only the verify call reads, are copied on a second stream once the draft
    logits are in, so that their transfer overlaps the tree build and the
    attention."""
    pin = {n: step.attn_h[n].pin_memory() for n in ("q", "tree_k", "tree_v")}
    draft_p = step.draft_h.pin_memory()
    target_p = step.target_h.pin_memory()
    out_acc = torch.empty(step.acc.numel() + 2, dtype=torch.int32).pin_memory()
    s2 = torch.cuda.Stream(device=s.device)
    times = []
    evs = []
    for _ in range(K):
        with torch.cuda.stream(s):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            drafted = torch.cuda.Event()
            e0.record(s)
            step.draft.copy_(draft_p, non_blocking=True)
            drafted.record(s)
        s2.wait_event(drafted)
        with torch.cuda.stream(s2):
            step.target.copy_(target_p, non_blocking=True)
            targeted = torch.cuda.Event()
            targeted.record(s2)
        with torch.cuda.stream(s):
            for n in ("q", "tree_k", "tree_v"):
                step.attn[n].copy_(pin[n], non_blocking=True)
            step.build(s)
            step.attention(s)
            s.wait_event(targeted)
            step.verify(s)
            out_acc[: step.acc.numel()].copy_(step.acc, non_blocking=True)
            out_acc[-2:-1].copy_(step.n_acc, non_blocking=True)
            out_acc[-1:].copy_(step.bonus, non_blocking=True)
            e1.record(s)
            evs.append((e0, e1))
    s.synchronize()
    s2.synchronize()
    for e0, e1 in evs:
        times.append(e0.elapsed_time(e1) * 1e3)
    d2h = (step.acc.numel() + 2) * 4
    return times, d2h


def spread(times):
    """p10 / median / p90 of per-step times (nearest-rank percentiles)."""
    xs = sorted(float(t) for t in times)
    if not xs:
        return None

    def rank(q):
        return round(xs[min(len(xs) - 1, max(0, -(-q * len(xs) // 100) - 1))], 3)

    return {"p10": rank(10), "median": round(statistics.median(xs), 3), "p90": rank(90)}


def max_over_ranks(x, world, device):
    """Slowest replica's value: the job's step time is set by the last rank
    to finish (all ranks run the same workload on their own GPU)."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# known ncu DRAM traffic per launch (bytes), keyed by kernel and source hash;
# entries whose hash no longer matches the sources are reported as null
TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one launch on the c2
    # workload from one ncu capture, keyed by the kernel's source hash
    # (_kernel_source_hash)
    "build:c2": ("c75e3b8f121a", 31664128),
    "verify:c2": ("7c14c3a06102", 36639232),
    "attn:c2": ("8e891d4a011d", 17385472),
}


def run_ours(args, rank, world, local_rank):
    import torch
    from eagle_speculative_decoding_verify_gb300 import _build
    _build.build()
    from eagle_speculative_decoding_verify_gb300 import binding as eb
    from eagle_speculative_decoding_verify_gb300 import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    step = Step(w, dev, eb, wl)
    s = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)
    with torch.cuda.stream(s):
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            step.run(s)
    s.synchronize()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local_rank] if vis else local_rank)
    sampler.start()
    time.sleep(0.15)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    try:
        times, _ = _time_graph(torch, step, s, flush, args.steps)
        graphed = True
    except Exception as exc:  # capture refused: time the plain stream launches
        print(f"cuda graph capture failed ({exc}); timing without a graph", file=sys.stderr)
        torch.cuda.synchronize()
        per0 = _time_kernels(torch, step, s, flush, args.steps)
        times = [a + b + c for a, b, c in zip(per0["build"], per0["attn"], per0["verify"])]
        graphed = False
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    sampler.window = (t_wall0, t_wall1)
    per = _time_kernels(torch, step, s, flush, args.steps)
    e2e_times, d2h = _time_e2e(torch, step, s, flush, args.steps)
    time.sleep(0.1)
    sampler.stop()

    us = max_over_ranks(statistics.mean(times), world, dev)
    hbm, tf, tf_sus, peak_src = _peaks()
    k_us = {k: statistics.mean(v) for k, v in per.items()}
    attn_gbs = step.bytes_attn() / (k_us["attn"] * 1e-6) / 1e9
    attn_tflops = step.flops_attn() / (k_us["attn"] * 1e-6) / 1e12
    dominant = max(k_us, key=k_us.get)
    if dominant == "attn" and step.flops_attn() / step.bytes_attn() > tf * 1e12 / (hbm * 1e9):
        roof = {"bound": "tensor", "achieved": attn_tflops, "peak": tf, "unit": "TFLOP/s",
                "frac": attn_tflops / tf}
    else:
        b = {"build": step.bytes_build(), "attn": step.bytes_attn(),
             "verify": step.bytes_verify()}[dominant]
        gbs = b / (k_us[dominant] * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm}
    tr = TRAFFIC.get(f"{dominant}:{args.workload}")
    roof.update({"kernel": dominant, "peak_source": peak_src,
                 "traffic": tr[1] if tr and tr[0] == _kernel_source_hash(dominant) else None})
    step_roof_us = (step.bytes_build() / (hbm * 1e3) + step.bytes_verify() / (hbm * 1e3) +
                    max(step.bytes_attn() / (hbm * 1e3), step.flops_attn() / (tf * 1e6)))
    line = {
        "metric": METRIC, "value": round(us, 3), "unit": "us", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "spread_us": spread(times),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 logits + bf16 attention (fp32 accumulate)" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded generators; no dataset or weights)",
        "config": {"workload": f"{args.workload} {WORKLOAD_LABEL[args.workload]}",
                   "l2": "flushed before every step (512 MB write, then 256 MB read)", "cuda_graph": graphed,
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "step_roofline_us": round(step_roof_us, 3),
        "step_roofline_frac": round(step_roof_us / us, 4),
        "kernels_us": {k: round(v, 3) for k, v in k_us.items()},
        "step_us_no_graph": round(sum(k_us.values()), 3),
        "tree_attn": {"achieved_gbs": round(attn_gbs, 1), "frac_hbm": round(attn_gbs / hbm, 4),
                      "achieved_tflops": round(attn_tflops, 1),
                      "frac_tensor": round(attn_tflops / tf, 4), "peak_source": peak_src},
        "e2e": {"value": round(statistics.mean(e2e_times), 3), "unit": "us",
                "h2d_bytes_per_step": step.h2d_bytes(), "d2h_bytes_per_step": d2h},
        "gpu_launches": step.launches * args.steps,
        "clocks": sampler.summary(),
    }
    with torch.cuda.stream(s):
        line["kv_commit"] = kv_commit_bench(eb, wl, dev, step, s)
        line["tree_expand"] = tree_expand_bench(eb, wl, dev, step, s, flush)
        line["tree_policy"] = tree_policy_bench(eb, wl, dev, step, s, flush)
        line["verify_nucleus"] = verify_nucleus_bench(eb, wl, dev, step, s, flush)
    if not args.no_long_attn:
        la = attn_long(eb, wl, dev)
        la["frac_hbm"] = round(la["achieved_gbs"] / hbm, 4)
        la["frac_tensor"] = round(la["achieved_tflops"] / tf, 4)
        if "fp8" in la:
            la["fp8"]["frac_hbm"] = round(la["fp8"]["achieved_gbs"] / hbm, 4)
            la["fp8"]["frac_tensor"] = round(la["fp8"]["achieved_tflops"] / tf, 4)
        la["peak_source"] = peak_src
        line["tree_attn_long"] = la
    if not args.no_configs:
        K = min(args.steps, 50)
        line["configs"] = {key: config_bench(eb, wl, dev, key, flush, K)
                           for key in ("c0", "c1", "c3", "c4")}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, samples=1)
        line["cpu_baseline_1thread_us"] = {key: oracle_one_thread(key).get("value")
                                           for key in ("c0", "c1", "c2")}
    return line


# ------------------------------------------------------------- oracle (CPU)
def _oracle_step(w, wl, inputs):
    from oracle.tree_attn import tree_attention
    from oracle.tree_build import build_draft_tree
    from oracle.verify import verify_tree
    draft, attn, root = inputs
    t = build_draft_tree(draft, w.top_k, w.depth, w.total_tokens, root)
    target = wl.target_logits(w, t["parents"], t["tokens"]).numpy()   # input generation
    t0 = time.perf_counter()
    tree_attention(*(attn[n] for n in NAMES), t["mask"], w.prefix)
    gr, T, k, p = w.sampling_of(0)
    verify_tree(target, t["parents"], t["tokens"], greedy=bool(gr), temperature=T, top_k=k,
                top_p=p, seed=1234, step=0)
    return time.perf_counter() - t0


def _oracle_inputs(w, wl):
    a = wl.attention_inputs(w)
    return (wl.draft_logits(w).numpy(), {n: a[n].double().numpy() for n in NAMES},
            wl.root_token(w))


def cpu_baseline(key, samples=1):
    """Oracle step time on the host cores (build + attention + verify; the
    target-logit generation between build and verify is not timed)."""
    from oracle.tree_build import build_draft_tree
    from eagle_speculative_decoding_verify_gb300 import workloads as wl
    w = wl.WORKLOADS[key]
    inputs = _oracle_inputs(w, wl)
    ts = []
    for _ in range(samples):
        t0 = time.perf_counter()
        build_draft_tree(inputs[0], w.top_k, w.depth, w.total_tokens, inputs[2])
        tb = time.perf_counter() - t0
        ts.append(tb + _oracle_step(w, wl, inputs))
    return {"value": round(statistics.mean(ts) * 1e6, 1), "unit": "us", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{samples} full step(s) of workload {key}: fp64 numpy tree build, "
                      "tree attention, acceptance walk"}


def run_reference(args):
    from eagle_speculative_decoding_verify_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    inputs = _oracle_inputs(w, wl)
    from oracle.tree_build import build_draft_tree

    def one():
        t0 = time.perf_counter()
        build_draft_tree(inputs[0], w.top_k, w.depth, w.total_tokens, inputs[2])
        return time.perf_counter() - t0 + _oracle_step(w, wl, inputs)

    for _ in range(min(args.warmup, 1)):
        one()
    budget = 150.0
    ts = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        ts.append(one())
        if time.perf_counter() - t_start > budget:
            break
    us = statistics.mean(ts) * 1e6
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us",
        "n_gpus": 0, "steps": len(ts), "warmup": args.warmup, "ms_per_step": us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators; no dataset or weights)",
        "config": {"workload": f"{args.workload} {WORKLOAD_LABEL[args.workload]}"},
        "cpu_baseline": {"value": round(us, 1), "unit": "us", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{len(ts)} full oracle step(s) of workload {args.workload} "
                                   "(timed steps capped at 150 s of host time)"},
        "e2e": {"value": round(us, 1), "unit": "us", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def profile_calls(case):
    """Three untimed iterations of one workload's library calls (a case for
    a profiler's launch filter)."""
    import torch
    from eagle_speculative_decoding_verify_gb300 import _build
    _build.build()
    from eagle_speculative_decoding_verify_gb300 import binding as eb, workloads as wl
    dev = torch.device("cuda")
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        if case == "c4":
            st = MultiStep(wl.WORKLOADS["c4"], dev, eb, wl)
            for _ in range(3):
                st.run(s)
        elif case in ("policy", "kv"):
            st = Step(wl.WORKLOADS["c2"], dev, eb, wl)
            if case == "policy":
                tree_policy_bench(eb, wl, dev, st, s, L2Flush(dev), reps=2)
            else:
                kv_commit_bench(eb, wl, dev, st, s, reps=3)
        else:
            st = Step(wl.WORKLOADS[case], dev, eb, wl)
            for _ in range(3):
                st.run(s)
    s.synchronize()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2", choices=["c0", "c1", "c2"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload step measurements of c0, c1, c3 and c4")
    ap.add_argument("--no-long-attn", action="store_true",
                    help="skip the 32-layer x 32K-context attention measurement")
    ap.add_argument("--long-attn-only", type=int, default=0, metavar="LAYERS",
                    help="only time the long-context attention, on LAYERS layers "
                         "(a profiling case; prints its own JSON line)")
    ap.add_argument("--fp8", action="store_true",
                    help="with --long-attn-only: also time the E4M3 prefix variant")
    ap.add_argument("--profile-calls", default="", metavar="CASE",
                    choices=["", "c0", "c1", "c2", "c4", "policy", "kv"],
                    help="run three untimed iterations of one workload's calls (c0-c2, c4: "
                         "build, attention, verify; policy: the tree policies on c2's draft "
                         "rows; kv: the KV commits) for a profiler, and print no JSON line")
    args = ap.parse_args()
    if args.profile_calls:
        return profile_calls(args.profile_calls)
    if args.long_attn_only:
        import torch
        from eagle_speculative_decoding_verify_gb300 import binding as eb, workloads as wl
        res = attn_long(eb, wl, torch.device("cuda"), reps=max(args.steps, 1),
                        n_layers=args.long_attn_only, paged=False, fp8=args.fp8)
        print(json.dumps(res), flush=True)
        return 0
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
