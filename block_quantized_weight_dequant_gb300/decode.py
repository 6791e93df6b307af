"""The GEMV weight stream of one batch-1 decode step.

A decoder layer's weight stream, in model order (RunIT README, data-flow
diagram: RMSNorm -> Q/K/V projections -> attention -> FFN gate/up -> SiLU ->
down -> ... -> lm_head):

    stage 4l+0: q, k, v        x = the layer input h
    stage 4l+1: o              x = q's output (stand-in for the attention
                               output, which has q's width)
    stage 4l+2: gate+up+SiLU   x = o's output, RMSNorm-ed with the layer gain
    stage 4l+3: down           x = the gate+up output; its output is the next
                               layer's input h
    last stage: LM head        x = the last layer's output

Attention itself, residual adds and the other norms are outside this stream
(they are not weight streaming).  Every op reads the previous stage's output,
so the stages are truly dependent, as in decode.  ``run_plan()`` runs the
stream through a plan (bq_stream_plan_*): one streaming-kernel launch per
stage, each waiting for the stage before (programmatic dependent launch; the
cooperative executor in one launch is the alternative); ``run_per_op()``
launches one kernel per op in stage order; the two give identical bits.

With ``chained=False`` every op instead reads an input vector of its own (the
same shapes and weights, no data flowing between ops): the pure per-token
weight stream, which a plan runs as ONE launch of the streaming kernel.

With ``fused_qkv=True`` each layer's q, k and v run as ONE op over their
rows concatenated at load time (``layer["qkv"]``, see ``concat_packed``)
with an optional fp32 bias (``layer["qkv_bias"]``): the fused QKV+bias
projection of the RunIT README (6 dispatches -> 1 per layer on the Qwen
path).  The op's output holds q, k and v back to back; o reads its q part.
"""
import torch

from . import StreamOp, StreamPlan, gemv, gemv_gate_up_silu, gemv_qkv_bias


class DecodeStream:
    def __init__(self, qtype, layers, lm_head, eps=1e-6, chained=True, fused_qkv=False):
        """layers: list of dicts with packed q, k, v, o, gate, up, down
        (uint8 [M, row bytes]) and gamma (fp32 [hidden]); with fused_qkv,
        packed qkv (the q, k, v rows concatenated) and optional qkv_bias
        (fp32) instead of q, k, v; lm_head: packed."""
        from . import _packed_shape, _qt
        self.qtype = _qt(qtype)
        self.eps = eps
        dev = lm_head.device
        self.layers = layers
        self.lm_head = lm_head
        f32 = dict(dtype=torch.float32, device=dev)

        def rows(P):
            return _packed_shape(P, self.qtype)

        hidden = rows(layers[0]["qkv" if fused_qkv else "q"])[1]
        self.fused_qkv = fused_qkv
        self.chained = chained
        # every vector the stream reads from outside lives in one buffer, so a
        # caller fills them with a single copy: x0 (chained), or x0 and one
        # input per op (unchained)
        n_in = hidden
        if not chained:
            for L in layers:
                n_in += rows(L["o"])[1] + hidden + rows(L["down"])[1] + hidden
        self.inputs = torch.zeros(n_in, **f32)
        self.x0 = self.inputs[:hidden]
        # likewise every op's output is a slice of one buffer, so a caller
        # reads them all back with a single copy; each slice starts on 16
        # bytes, as an output that a later stage reads as its x must
        def pad4(n):
            return (n + 3) // 4 * 4

        n_out = pad4(rows(lm_head)[0])
        for L in layers:
            n_out += sum(pad4(rows(L[n])[0]) for n in (("qkv",) if fused_qkv else ("q", "k", "v")))
            n_out += pad4(rows(L["o"])[0]) + pad4(rows(L["gate"])[0]) + pad4(rows(L["down"])[0])
        self.outputs = torch.zeros(n_out, **f32)
        ocursor = [0]

        def out(n):
            t = self.outputs[ocursor[0]:ocursor[0] + n]
            ocursor[0] += pad4(n)
            return t

        self.ops = []
        self.buffers = []
        cursor = [hidden]

        def src(produced, K):
            # chained: the producing op's output; otherwise an input of its own
            if chained:
                return produced
            t = self.inputs[cursor[0]:cursor[0] + K]
            cursor[0] += K
            return t

        h = self.x0
        st = 0
        for L in layers:
            q_dim = rows(L["o"])[1]  # o reads the attention output, q's width
            bufs = {}
            if fused_qkv:
                bufs["qkv"] = out(rows(L["qkv"])[0])
                bufs["q"] = bufs["qkv"][:q_dim]
                self.ops.append(StreamOp(st, L["qkv"], h, bufs["qkv"], bias=L.get("qkv_bias")))
            else:
                for n in ("q", "k", "v"):
                    bufs[n] = out(rows(L[n])[0])
                    self.ops.append(StreamOp(st, L[n], h, bufs[n]))
            bufs["o"] = out(rows(L["o"])[0])
            bufs["ffn"] = out(rows(L["gate"])[0])
            bufs["down"] = out(rows(L["down"])[0])
            self.buffers.append(bufs)
            self.ops.append(StreamOp(st + 1, L["o"], src(bufs["q"], q_dim), bufs["o"]))
            self.ops.append(StreamOp(st + 2, L["gate"], src(bufs["o"], hidden), bufs["ffn"],
                                     W_up=L["up"], gamma=L["gamma"], eps=eps))
            self.ops.append(StreamOp(st + 3, L["down"], src(bufs["ffn"], rows(L["down"])[1]),
                                     bufs["down"]))
            h = src(bufs["down"], hidden)
            st += 4
        self.logits = out(rows(lm_head)[0])
        assert ocursor[0] == n_out
        self.ops.append(StreamOp(st, lm_head, h, self.logits))
        self._plan = None

    @property
    def n_stages(self):
        return self.ops[-1].stage + 1

    def weight_bytes(self):
        n = 0
        for op in self.ops:
            n += op.W.numel() + (op.W_up.numel() if op.W_up is not None else 0)
        return n

    def activation_bytes(self):
        """Algorithmic activation traffic: every op reads x (and gamma or
        bias) and writes y once."""
        n = 0
        for op in self.ops:
            n += 4 * (op.x.numel() + op.y.numel())
            if op.gamma is not None:
                n += 4 * op.gamma.numel()
            if op.bias is not None:
                n += 4 * op.bias.numel()
        return n

    def plan(self):
        if self._plan is None:
            self._plan = StreamPlan(self.qtype, self.ops)
        return self._plan

    def run_plan(self):
        self.plan().launch()

    def run_per_op(self):
        for op in self.ops:
            if op.W_up is None and op.bias is not None:
                gemv_qkv_bias(self.qtype, op.W, op.x, op.bias, op.y)
            elif op.W_up is None:
                gemv(self.qtype, op.W, op.x, op.y)
            else:
                gemv_gate_up_silu(self.qtype, op.W, op.W_up, op.x, op.gamma, op.eps, op.y)
