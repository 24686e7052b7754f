"""A random-init Qwen3-8B-shaped decoder served with continuous batching on the
batch-invariant kernels.

Every reduction of the forward pass runs in this library's kernels (RMSNorm,
GEMM, prefill and decode attention), and so do the per-token steps around
them (per-head q/k norm + RoPE + paged KV append, SwiGLU, residual add fused
with RMSNorm).  The only torch operations are the embedding-row gather and the
final argmax, both exact.  So a request's logits are bit-identical whatever
else shares its step -- the property "Defeating Nondeterminism in LLM
Inference: The Core Role of Batch Invariance" ("Experimental Validation")
demonstrates end to end, here on random weights instead of a trained model.

Scheduler: each step takes every running sequence's next token (decode), then
fills the rest of a per-step token budget with prompt tokens of waiting
sequences -- a prompt that does not fit is split across steps (chunked
prefill).  Decode rows use bi_decode_attention; prompt rows use
bi_prefill_attention; both give a token the same bits.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch

from . import (add_rmsnorm, decode_attention, decode_attention_workspace_size, gemm,
               gemm_swiglu, interleave_gate_up, logprobs, prefill_attention,
               prefill_attention_workspace_size, qk_norm_rope_append, rmsnorm, silu_mul)
from . import inputs
from ._lib import PAGE_SIZE


def rope_table(max_pos: int, theta: float, D: int = 128, device=None) -> torch.Tensor:
    """The model's RoPE table, an input of bi_qk_norm_rope_append like a
    weight: fp32 [max_pos][D] with cos(pos * f_i) at i and sin(pos * f_i) at
    D/2 + i, f_i = theta^(-i/(D/2)) (rotate-half pairing), evaluated in float64
    on the host and rounded once to fp32."""
    half = D // 2
    pos = torch.arange(max_pos, dtype=torch.float64)[:, None]
    f = torch.pow(torch.tensor(float(theta), dtype=torch.float64),
                  -torch.arange(half, dtype=torch.float64) / half)[None, :]
    ang = pos * f
    tab = torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32)
    return tab.to(device) if device is not None else tab


@dataclass
class Qwen3Config:
    hidden: int = 4096
    layers: int = 36
    ffn: int = 12288
    heads: int = 32
    kv_heads: int = 8
    head_dim: int = 128
    vocab: int = 151936
    rope_theta: float = 1e6
    eps: float = 1e-6
    max_pos: int = 8192


class Qwen3Weights:
    """Seeded random-init weights on the device: linear layers ~ N(0, 0.02)
    in the nn.Linear [out, in] layout, norm weights 1 (q/k norms included),
    untied embedding and lm_head."""

    def __init__(self, cfg: Qwen3Config, seed: int = 1000, device="cuda"):
        self.cfg = cfg
        H, F, D = cfg.hidden, cfg.ffn, cfg.head_dim
        qkv_out = (cfg.heads + 2 * cfg.kv_heads) * D
        w = lambda shape, k: inputs.normal_bf16(shape, seed + k, std=0.02, device=device)  # noqa: E731
        ones = lambda n: torch.ones(n, dtype=torch.bfloat16, device=device)  # noqa: E731
        self.embed = w((cfg.vocab, H), 0)
        self.lm_head = w((cfg.vocab, H), 1)
        self.final_norm = ones(H)
        self.layers = []
        for l in range(cfg.layers):
            b = 10 + 10 * l
            self.layers.append({
                "in_norm": ones(H), "qkv": w((qkv_out, H), b), "q_norm": ones(D),
                "k_norm": ones(D), "o": w((H, cfg.heads * D), b + 1), "post_norm": ones(H),
                "gate_up": w((2 * F, H), b + 2), "down": w((H, F), b + 3)})

    def host_bits(self, n_layers: int) -> dict:
        """uint16 bit patterns of the first n_layers layers (for the oracle)."""
        def b(t):
            return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        out = {"embed": b(self.embed), "lm_head": b(self.lm_head),
               "final_norm": b(self.final_norm)}
        for l in range(n_layers):
            for k, v in self.layers[l].items():
                out[f"{l}.{k}"] = b(v)
        return out


@dataclass
class Sequence:
    sid: int
    prompt: list
    max_new: int
    generated: list = field(default_factory=list)
    forced: list | None = None  # teacher-forced continuation instead of argmax
    n_cached: int = 0
    pages: list = field(default_factory=list)

    @property
    def tokens(self):
        return self.prompt + self.generated

    @property
    def done(self):
        return len(self.generated) >= self.max_new


class Engine:
    """Paged KV cache + continuous-batching greedy decode over Qwen3Weights
    (optionally truncated to the first n_layers layers)."""

    GRAPH_BUCKETS = (1, 2, 4, 8, 16, 32, 64, 128, 256)

    def __init__(self, weights: Qwen3Weights, num_pages: int, max_tokens_per_step: int = 8192,
                 n_layers: int | None = None, device="cuda", ops: str = "bi",
                 cuda_graphs: bool = False):
        """ops="bi": every GEMM and RMSNorm through this library (batch-invariant).
        ops="torch": GEMMs through torch.matmul (cuBLAS) and RMSNorms through
        torch.nn.functional.rms_norm instead -- the non-invariant comparison.
        cuda_graphs: run decode-only steps of up to 256 sequences as a CUDA
        graph captured once per batch bucket (1, 2, 4, ... 256 rows), padded
        with rows that read and write one reserved page.  The kernels are the
        same, and no row's arithmetic depends on the others, so the logits are
        the same bits as without graphs; what goes away is the per-launch host
        work of about 300 launches a step."""
        if ops not in ("bi", "torch"):
            raise ValueError("ops must be 'bi' or 'torch'")
        self.ops = ops
        self.w = weights
        cfg = self.cfg = weights.cfg
        self.n_layers = n_layers or cfg.layers
        self.device = torch.device(device)
        self.num_pages = num_pages
        self.budget = max_tokens_per_step
        D, Hkv = cfg.head_dim, cfg.kv_heads
        self.k_cache = [torch.empty(num_pages, Hkv, PAGE_SIZE, D, dtype=torch.bfloat16,
                                    device=self.device) for _ in range(self.n_layers)]
        self.v_cache = [torch.empty_like(k) for k in self.k_cache]
        self.cuda_graphs = cuda_graphs
        if cuda_graphs and num_pages < 2:
            raise ValueError("cuda_graphs needs a spare page for padding rows")
        # with graphs, the last page belongs to the padding rows
        self.pad_page = num_pages - 1 if cuda_graphs else None
        self.free_pages = deque(range(num_pages - 1 if cuda_graphs else num_pages))
        self._graphs = {}
        self._ws = None
        self._pws = None
        self.graph_steps = 0
        self.rope = rope_table(cfg.max_pos, cfg.rope_theta, D, device=self.device)
        T, H, F = max_tokens_per_step, cfg.hidden, cfg.ffn
        e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=self.device)  # noqa: E731
        self.buf = {"res": e(T, H), "n": e(T, H), "qkv": e(T, (cfg.heads + 2 * Hkv) * D),
                    "q": e(T, cfg.heads, D), "attn": e(T, cfg.heads, D), "o": e(T, H),
                    "gu": e(T, 2 * F), "h": e(T, F), "d": e(T, H)}
        # the bi path runs gate|up and SwiGLU as one fused GEMM over an
        # interleaved copy of the weight (bit-identical to gemm + silu_mul)
        self.gate_up_il = ([interleave_gate_up(self.w.layers[l]["gate_up"])
                            for l in range(self.n_layers)] if ops == "bi" else None)
        self.steps = 0

    # ------------------------------------------------------------ pages ----
    def _ensure_pages(self, seq: Sequence, upto: int):
        need = -(-upto // PAGE_SIZE)
        while len(seq.pages) < need:
            if not self.free_pages:
                raise RuntimeError("KV cache out of pages")
            seq.pages.append(self.free_pages.popleft())

    def _release(self, seq: Sequence):
        self.free_pages.extend(seq.pages)
        seq.pages = []

    # ---------------------------------------------------------- forward ----
    def forward(self, items, want_logits, pending=None):
        """One step.  items: list of (seq, n) -- process the next n uncached
        tokens of seq.  want_logits: per item, whether its last token's logits
        are needed.  pending: None, or (picks, {id(seq): j}) for decode items
        whose input token is the previous step's pick still on the device
        (picks[j]).  Returns logits [sum(want_logits), vocab] (bf16) or None.
        Nothing here waits for the device: step metadata goes up from pinned
        host memory behind the work already queued."""
        cfg = self.cfg
        dev = self.device
        toks, pos, slots = [], [], []
        fill_rows, fill_src = [], []
        src_of = pending[1] if pending is not None else {}
        for seq, n in items:
            t0 = seq.n_cached
            self._ensure_pages(seq, t0 + n)
            if n == 1:
                j = src_of.get(id(seq))
                if j is not None:
                    fill_rows.append(len(toks))
                    fill_src.append(j)
                    toks.append(0)
                else:
                    toks.append(seq.tokens[t0])
                pos.append(t0)
                slots.append(seq.pages[t0 // PAGE_SIZE] * PAGE_SIZE + t0 % PAGE_SIZE)
            else:
                tt = np.arange(t0, t0 + n)
                toks.extend(seq.tokens[t0:t0 + n])
                pos.extend(range(t0, t0 + n))
                slots.extend((np.asarray(seq.pages)[tt // PAGE_SIZE] * PAGE_SIZE
                              + tt % PAGE_SIZE).tolist())
        T = len(toks)
        if T > self.budget:
            raise ValueError("step exceeds the token budget")

        def up(a, dtype):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=dtype)).pin_memory().to(
                dev, non_blocking=True)
        i32 = lambda a: up(a, np.int32)  # noqa: E731
        tok_d = up(toks, np.int64)
        if fill_rows:
            tok_d[up(fill_rows, np.int64)] = pending[0][up(fill_src, np.int64)]
        pos_d, slot_d = i32(pos), i32(slots)

        # decode items (one token) and prompt items, each with its own metadata
        dec = [(k, s, n) for k, (s, n) in enumerate(items) if n == 1 and s.n_cached >= len(s.prompt)]
        pre = [(k, s, n) for k, (s, n) in enumerate(items) if not (n == 1 and s.n_cached >= len(s.prompt))]
        offs = np.cumsum([0] + [n for _, n in items])

        def table(group):
            width = max(len(s.pages) for _, s, _ in group)
            bt = np.full((len(group), width), -1, dtype=np.int32)
            for r, (_, s, _) in enumerate(group):
                bt[r, :len(s.pages)] = s.pages
            return bt

        meta = {}
        if dec:
            rows = np.array([offs[k] for k, _, _ in dec], dtype=np.int64)
            lens = [s.n_cached + 1 for _, s, _ in dec]
            bt = table(dec)
            meta["dec"] = (self._rows(rows, up), i32(bt), i32(lens), int(max(lens)), bt.shape[1])
            meta["ws"] = self._att_workspace(len(dec), int(max(lens)))
        if pre:
            starts = [int(offs[k]) for k, _, _ in pre]
            nqs = [n for _, _, n in pre]
            # prompt rows are contiguous per item; gather them into one block
            rows = np.concatenate([np.arange(a, a + n) for a, n in zip(starts, nqs)])
            indptr = np.concatenate([[0], np.cumsum(nqs)])
            lens = [s.n_cached + n for _, s, n in pre]
            bt = table(pre)
            meta["pre"] = (self._rows(rows, up), i32(bt), i32(lens), i32(indptr),
                           int(max(nqs)), int(max(lens)))
            meta["pws"] = self._prefill_workspace(len(rows), int(max(lens)))

        b = {k: v[:T] for k, v in self.buf.items()}
        self._layers(b, T, tok_d, pos_d, slot_d, meta)
        samp = [int(offs[k + 1] - 1) for k, want in enumerate(want_logits) if want]
        if not samp:
            return None
        nrows = torch.index_select(b["n"], 0, up(samp, np.int64))
        self.steps += 1
        return gemm(nrows, self.w.lm_head, out=torch.empty(len(samp), cfg.vocab,
                                                           dtype=torch.bfloat16, device=dev))

    def _layers(self, b, T, tok_d, pos_d, slot_d, meta):
        """Embedding, every decoder layer and the final norm for the step's T
        token rows (into b["n"])."""
        cfg = self.cfg
        res = b["res"]
        gemm, rmsnorm, add_rmsnorm = self._ops()
        torch.index_select(self.w.embed, 0, tok_d, out=res)
        Hq, Hkv = cfg.heads, cfg.kv_heads
        for l in range(self.n_layers):
            L = self.w.layers[l]
            if l == 0:
                rmsnorm(res, L["in_norm"], cfg.eps, out=b["n"])
            else:
                add_rmsnorm(b["d"], res, L["in_norm"], cfg.eps, out=b["n"])
            gemm(b["n"], L["qkv"], out=b["qkv"])
            qk_norm_rope_append(b["qkv"], Hq, Hkv, pos_d, slot_d, self.rope, L["q_norm"],
                                L["k_norm"], self.k_cache[l], self.v_cache[l], cfg.eps,
                                q_out=b["q"])
            self._attention(l, b, meta)
            gemm(b["attn"].view(T, Hq * cfg.head_dim), L["o"], out=b["o"])
            add_rmsnorm(b["o"], res, L["post_norm"], cfg.eps, out=b["n"])
            if self.gate_up_il is not None:
                gemm_swiglu(b["n"], self.gate_up_il[l], out=b["h"])
            else:
                gemm(b["n"], L["gate_up"], out=b["gu"])
                silu_mul(b["gu"], out=b["h"])
            gemm(b["h"], L["down"], out=b["d"])
        add_rmsnorm(b["d"], res, self.w.final_norm, cfg.eps, out=b["n"])

    # ----------------------------------------------------------- graphs ----
    def _graph_for(self, Bb: int):
        """The captured decode step for Bb rows, with its static inputs."""
        if Bb in self._graphs:
            return self._graphs[Bb]
        cfg, dev = self.cfg, self.device
        W = cfg.max_pos // PAGE_SIZE
        i32 = dict(dtype=torch.int32, device=dev)
        st = {"tok": torch.zeros(Bb, dtype=torch.int64, device=dev),
              "pos": torch.zeros(Bb, **i32),
              "slot": torch.full((Bb,), self.pad_page * PAGE_SIZE, **i32),
              "lens": torch.ones(Bb, **i32),
              "bt": torch.full((Bb, W), self.pad_page, **i32),
              "logits": torch.empty(Bb, cfg.vocab, dtype=torch.bfloat16, device=dev),
              # zero-filled: its leading arrival counters must start at zero
              "ws": torch.zeros(decode_attention_workspace_size(Bb, cfg.heads, cfg.head_dim,
                                                                cfg.max_pos),
                                dtype=torch.uint8, device=dev)}
        meta = {"dec": (slice(0, Bb), st["bt"], st["lens"], cfg.max_pos, W), "ws": st["ws"]}
        b = {k: v[:Bb] for k, v in self.buf.items()}
        gemm_, _, _ = self._ops()

        def body():
            self._layers(b, Bb, st["tok"], st["pos"], st["slot"], meta)
            gemm_(b["n"], self.w.lm_head, out=st["logits"])

        # one eager run first (library set-up happens outside the capture)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            body()
        torch.cuda.current_stream(dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()
        self._graphs[Bb] = (g, st)
        return self._graphs[Bb]

    def _graph_step(self, items, pending):
        """A decode-only step through the captured graph of its bucket.
        Returns logits [len(items), vocab] (valid until the next replay)."""
        B = len(items)
        Bb = next(x for x in self.GRAPH_BUCKETS if x >= B)
        g, st = self._graph_for(Bb)
        W = st["bt"].shape[1]
        tok = np.zeros(Bb, dtype=np.int64)
        pos = np.zeros(Bb, dtype=np.int32)
        slot = np.full(Bb, self.pad_page * PAGE_SIZE, dtype=np.int32)
        lens = np.ones(Bb, dtype=np.int32)
        bt = np.full((Bb, W), self.pad_page, dtype=np.int32)
        fill_rows, fill_src = [], []
        src_of = pending[1] if pending is not None else {}
        for r, (seq, _) in enumerate(items):
            t0 = seq.n_cached
            self._ensure_pages(seq, t0 + 1)
            j = src_of.get(id(seq))
            if j is not None:
                fill_rows.append(r)
                fill_src.append(j)
            else:
                tok[r] = seq.tokens[t0]
            pos[r] = t0
            slot[r] = seq.pages[t0 // PAGE_SIZE] * PAGE_SIZE + t0 % PAGE_SIZE
            lens[r] = t0 + 1
            bt[r, :len(seq.pages)] = seq.pages
        for name, arr in (("tok", tok), ("pos", pos), ("slot", slot), ("lens", lens), ("bt", bt)):
            st[name].copy_(torch.from_numpy(arr).pin_memory(), non_blocking=True)
        if fill_rows:
            idx = torch.from_numpy(np.asarray(fill_rows, dtype=np.int64)).pin_memory().to(
                self.device, non_blocking=True)
            src = torch.from_numpy(np.asarray(fill_src, dtype=np.int64)).pin_memory().to(
                self.device, non_blocking=True)
            st["tok"][idx] = pending[0][src]
        g.replay()
        self.steps += 1
        self.graph_steps += 1
        return st["logits"][:B]

    def _att_workspace(self, B: int, max_len: int):
        """The eager steps' decode-attention workspace, kept across steps and
        grown when a step needs more.  It is zero-filled when allocated: its
        leading arrival counters must start at zero, and every call leaves
        them zero, so it is never cleared again."""
        cfg = self.cfg
        need = decode_attention_workspace_size(B, cfg.heads, cfg.head_dim, max_len)
        if need == 0:
            return None
        if self._ws is None or self._ws.numel() < need:
            self._ws = None
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def _prefill_workspace(self, T: int, max_len: int):
        """The prefill-attention workspace (running output of prompt rows
        longer than one 256-token chunk), kept across steps and grown when a
        step needs more; its contents need no initialisation."""
        cfg = self.cfg
        need = prefill_attention_workspace_size(T, cfg.heads, cfg.head_dim, max_len)
        if need == 0:
            return None
        if self._pws is None or self._pws.numel() < need:
            self._pws = None
            self._pws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._pws

    def _ops(self):
        if self.ops == "bi":
            return gemm, rmsnorm, add_rmsnorm
        import torch.nn.functional as F

        def t_gemm(x, W, out=None):
            return torch.matmul(x, W.t(), out=out)

        def t_rmsnorm(x, w, eps, out=None):
            out.copy_(F.rms_norm(x, (x.shape[-1],), w, eps))
            return out

        def t_add_rmsnorm(x, res, w, eps, out=None):
            res.add_(x)
            out.copy_(F.rms_norm(res, (res.shape[-1],), w, eps))
            return out
        return t_gemm, t_rmsnorm, t_add_rmsnorm

    @staticmethod
    def _rows(rows, up):
        """A group's token rows: a slice when they are one contiguous run (the
        scheduler puts decode rows first and prompt rows after them), else a
        device index tensor."""
        if len(rows) and rows[-1] - rows[0] + 1 == len(rows) and (np.diff(rows) == 1).all():
            return slice(int(rows[0]), int(rows[-1]) + 1)
        return up(rows, np.int64)

    def _attention(self, l, b, meta):
        kc, vc = self.k_cache[l], self.v_cache[l]
        for kind in ("dec", "pre"):
            if kind not in meta:
                continue
            rows = meta[kind][0]
            if isinstance(rows, slice):  # q rows and outputs in place
                q, out = b["q"][rows], b["attn"][rows]
            else:
                q, out = torch.index_select(b["q"], 0, rows), None
            if kind == "dec":
                _, bt, lens, mx, _ = meta[kind]
                out = decode_attention(q, kc, vc, bt, lens, max_seq_len=mx, out=out,
                                       workspace=meta.get("ws"))
            else:
                _, bt, lens, indptr, mq, mx = meta[kind]
                out = prefill_attention(q, kc, vc, bt, lens, indptr, max_q_len=mq,
                                        max_seq_len=mx, out=out, workspace=meta.get("pws"))
            if not isinstance(rows, slice):
                b["attn"].index_copy_(0, rows, out)

    # ------------------------------------------------------- scheduling ----
    def generate(self, seqs: list[Sequence], record: set | None = None):
        """Run every sequence to max_new generated tokens.  Returns
        {sid: [logits row per generated token]} (CPU bf16) for sids in `record`;
        the log-probability of each generated token (bi_logprobs, fp32) goes to
        self.logprobs[sid] for the same sids.

        The host runs one step ahead of the device: step i+1 is planned and
        queued while step i computes (no request ends early, so the schedule
        never needs a token's value), its decode rows take their input tokens
        straight from step i's picks on the device, and step i's picks are
        read back only after step i+1 has been queued."""
        record = record or set()
        rec_rows = {sid: [] for sid in record}  # device rows, copied to the host at the end
        waiting = deque(seqs)
        running: list[Sequence] = []
        prev = None
        while waiting or running:
            items, budget = [], self.budget
            for s in running:
                items.append((s, 1))
                budget -= 1
            admitted = []
            while waiting and budget > 0:
                s = waiting[0]
                take = min(len(s.prompt) - s.n_cached, budget)
                items.append((s, take))
                budget -= take
                if s.n_cached + take == len(s.prompt):
                    admitted.append(waiting.popleft())
                else:
                    break
            want = [s.n_cached + n == len(s.tokens) for s, n in items]
            decode_only = all(n == 1 and s.n_cached >= len(s.prompt) for s, n in items)
            if self.cuda_graphs and decode_only and 0 < len(items) <= self.GRAPH_BUCKETS[-1]:
                logits = self._graph_step(items, prev[:2] if prev else None)
            else:
                logits = self.forward(items, want, pending=prev[:2] if prev else None)
            if prev is not None:
                self._resolve(prev)
            prev = None
            for s, n in items:
                s.n_cached += n
            sampled = [s for (s, n), w in zip(items, want) if w]
            if logits is not None:
                picks = torch.argmax(logits, dim=-1)
                forced = [(j, s.forced[len(s.generated)]) for j, s in enumerate(sampled)
                          if s.forced is not None]
                if forced:
                    fj = self._up([j for j, _ in forced])
                    picks[fj] = self._up([v for _, v in forced])
                rec = [(j, s.sid) for j, s in enumerate(sampled) if s.sid in record]
                if rec:
                    rj = self._up([j for j, _ in rec])
                    lg = torch.index_select(logits, 0, rj)
                    lps, _ = logprobs(lg, picks[rj].to(torch.int32))
                    for i, (_, sid) in enumerate(rec):
                        rec_rows[sid].append((lg, lps, i))
                host = torch.empty(picks.shape, dtype=picks.dtype, pin_memory=True)
                host.copy_(picks, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record()
                slot_of = {}
                for j, s in enumerate(sampled):
                    slot_of[id(s)] = j
                    s.generated.append(None)  # filled in by _resolve
                prev = (picks, slot_of, host, ev, sampled)
            running = [s for s in running + admitted if not s.done]
            for s in seqs:
                if s.done and s.pages:
                    self._release(s)
        if prev is not None:
            self._resolve(prev)
        logs, self.logprobs = {}, {}
        for sid, rows in rec_rows.items():
            lg = torch.stack([t[i] for t, _, i in rows]).cpu() if rows else None
            lp = torch.stack([t[i] for _, t, i in rows]).cpu() if rows else None
            logs[sid] = list(lg.unbind(0)) if rows else []
            self.logprobs[sid] = list(lp.unbind(0)) if rows else []
        return logs

    def _up(self, values):
        """int64 host list -> device tensor through pinned memory, without
        waiting for the device (a plain torch.tensor(..., device=...) copy from
        pageable memory would stall the host until the stream drains)."""
        return torch.from_numpy(np.asarray(values, dtype=np.int64)).pin_memory().to(
            self.device, non_blocking=True)

    @staticmethod
    def _resolve(prev):
        """Wait for one step's picks to reach the host and store them."""
        _, _, host, ev, sampled = prev
        ev.synchronize()
        vals = host.tolist()
        for j, s in enumerate(sampled):
            # a step is resolved before the next one appends its placeholder,
            # so the step's pick is the last entry
            s.generated[-1] = int(vals[j])

    def reset(self):
        self.free_pages = deque(range(self.num_pages - 1 if self.cuda_graphs else self.num_pages))
        self.steps = 0
        self.graph_steps = 0


def random_requests(n: int, vocab: int, min_len: int, max_len: int, max_new: int,
                    seed: int = 7) -> list[Sequence]:
    """n requests with prompt lengths uniform on [min_len, max_len] and token
    ids uniform on [0, vocab)."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(min_len, max_len + 1, (n,), generator=g).tolist()
    out = []
    for i, L in enumerate(lens):
        prompt = torch.randint(0, vocab, (L,), generator=g).tolist()
        out.append(Sequence(sid=i, prompt=prompt, max_new=max_new))
    return out
