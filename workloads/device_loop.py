"""Closed-loop decode driver on the GPU (harness only).

Holds the device buffers of one workload and runs its decode steps through a
Graft engine object (anything with the ``assemble`` / ``verify_update`` /
``warmup`` methods of ``hybrid_draft_tree_gb300.Graft``): draft inputs are
generated on the host and copied in, the synthetic target's logits are filled
on the device from the assembled tree, and the request state advances on the
device from the accepted tokens.
"""
from __future__ import annotations

import numpy as np

from . import F32, MODE_TAIL, DeviceSynth, Harness, Workload


class DeviceLoop:
    def __init__(self, w: Workload, engine, device="cuda:0", stream=None, track_src=False):
        import torch
        self.torch = torch
        self.w = w
        self.g = engine
        self.device = torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.h = Harness(w)
        self.ds = DeviceSynth(self.h, self.device)
        B, S, n = w.B, w.S, w.draft_nodes
        dev = self.device
        root, prev, ctx = self.h.init_state()
        self.root_h, self.prev_h, self.ctx_h = root, prev, ctx
        self.root = torch.from_numpy(root).to(dev)
        self.prev = torch.from_numpy(prev).to(dev)
        self.ctx = torch.from_numpy(ctx.view(np.int64)).to(dev)
        self.d_tok = torch.empty((B, n), dtype=torch.int32, device=dev)
        self.d_par = torch.empty((B, n), dtype=torch.int16, device=dev)
        self.d_aux = torch.empty((B, n), dtype=torch.float32, device=dev)
        self.tok = torch.empty((B, S), dtype=torch.int32, device=dev)
        self.par = torch.empty((B, S), dtype=torch.int8, device=dev)
        self.pos = torch.empty((B, S), dtype=torch.int32, device=dev)
        self.mask = torch.empty((B, S), dtype=torch.int64, device=dev)
        self.info = torch.empty((B, 4), dtype=torch.int32, device=dev)
        # with track_src, assemble also writes each slot's provenance (0 root, 1 draft, 2 retrieved, -1 pad)
        self.src = torch.empty((B, S), dtype=torch.int8, device=dev) if track_src else None
        self.accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
        self.out_tokens = torch.empty((B, S), dtype=torch.int32, device=dev)
        ldt = torch.float32 if w.dtype == F32 else torch.bfloat16
        self.logits = torch.empty((B * S, w.V), dtype=ldt, device=dev)
        self.step_index = 0
        self.host_draft = None

    # --- per-step pieces ---------------------------------------------------------------
    def draft(self, step=None):
        """Generate this step's draft inputs on the host from the host state and
        copy them to the device (non-blocking from pinned memory)."""
        step = self.step_index if step is None else step
        tok, par, aux = self.h.draft(step, self.root_h, self.prev_h)
        self.host_draft = (tok, par, aux)
        with self.torch.cuda.stream(self.stream):
            self.d_tok.copy_(self.torch.from_numpy(tok))
            if par is not None:
                self.d_par.copy_(self.torch.from_numpy(par))
            self.d_aux.copy_(self.torch.from_numpy(aux))
        return tok, par, aux

    def assemble(self):
        par = None if self.w.mode == MODE_TAIL else self.d_par
        if self.src is None:
            self.g.assemble(self.w.B, self.root, self.d_tok, par, self.d_aux, self.tok, self.par, self.pos, self.mask,
                            self.info, stream=self.stream)
        else:
            self.g.assemble(self.w.B, self.root, self.d_tok, par, self.d_aux, self.tok, self.par, self.pos, self.mask,
                            self.info, stream=self.stream, slot_src=self.src)

    def assemble_incremental(self, side_stream=None):
        """The same step through the incremental-drafting calls: checkpoint
        verdicts layer by layer on growing prefixes of this step's draft (as
        a drafter would make them), the retrieval gather on `side_stream`, then
        the staged assembly.  Leaves the verdicts in self.event and the
        gathered entries in self.retrieved."""
        torch = self.torch
        B, n = self.w.B, self.w.draft_nodes
        if not hasattr(self, "event"):
            self.event = torch.empty((B,), dtype=torch.int32, device=self.device)
            self.retrieved = torch.empty((B, self.w.budget), dtype=torch.int32, device=self.device)
        par_h = self.host_draft[1][0]
        depth = np.zeros(n, np.int32)
        for i in range(n):
            depth[i] = 0 if par_h[i] < 0 else depth[par_h[i]] + 1
        with torch.cuda.stream(self.stream):
            self.event.fill_(-1)
            for L in range(int(depth.max()) + 1 if n else 0):
                m = int((depth <= L).sum())          # BFS order: layers 0..L are a prefix
                self.g.check(B, self.d_par[:, :m].contiguous(), self.d_aux[:, :m].contiguous(), L, self.event,
                             stream=self.stream)
        side = side_stream if side_stream is not None else self.stream
        side.wait_stream(self.stream)
        self.g.retrieve(B, self.root, self.event, self.retrieved, stream=side)
        self.stream.wait_stream(side)
        self.g.assemble_staged(B, self.root, self.d_tok, self.d_par, self.d_aux, self.event, self.retrieved, self.tok,
                               self.par, self.pos, self.mask, self.info, stream=self.stream)

    def make_logits(self):
        s = self.stream.cuda_stream
        rk, pl, bi = self.ds.tree_rowparams(self.tok, self.par, self.ctx, self.prev, s)
        self.ds.fill_rows(rk.view(-1), pl.view(-1), bi.view(-1), self.logits, s)

    def verify_update(self):
        self.g.verify_update(self.w.B, self.tok, self.par, self.pos, self.mask, self.logits, self.accept_len,
                             self.out_tokens, stream=self.stream)

    def advance(self, read_back=True):
        self.ds.advance(self.out_tokens, self.accept_len, self.root, self.prev, self.ctx, self.stream.cuda_stream)
        self.step_index += 1
        if read_back:
            self.pull_state()

    def pull_state(self):
        self.stream.synchronize()
        self.root_h = self.root.cpu().numpy()
        self.prev_h = self.prev.cpu().numpy()
        self.ctx_h = self.ctx.cpu().numpy().view(np.uint64)

    def step(self):
        self.draft()
        self.assemble()
        self.make_logits()
        self.verify_update()
        self.advance()

    # --- warm-up ---------------------------------------------------------------------------
    def warm_inputs_device(self, rows_per_chunk=None):
        """(tokens, logits) of the workload's warm-up on the device, or None."""
        wr = self.h.warm_rowparams()
        if wr is None:
            return None
        toks, rk, pl, bi = wr
        torch = self.torch
        dev = self.device
        ldt = torch.float32 if self.w.dtype == F32 else torch.bfloat16
        logits = torch.empty((len(toks), self.w.V), dtype=ldt, device=dev)
        with torch.cuda.stream(self.stream):
            rk_d = torch.from_numpy(rk.view(np.int64)).to(dev)
            pl_d = torch.from_numpy(pl).to(dev)
            bi_d = torch.from_numpy(bi).to(dev)
            self.ds.fill_rows(rk_d, pl_d, bi_d, logits, self.stream.cuda_stream)
            toks_d = torch.from_numpy(toks).to(dev)
        return toks_d, logits, (toks, rk, pl, bi)
