"""Shared helpers of the GPU parity tests: device model construction and the oracle's view
of the same synthetic inputs.  The oracle only ever receives generator outputs and the
GPU's own logits (for the decision protocol); no oracle input comes from GPU results
otherwise."""
from __future__ import annotations

import numpy as np

import oracle
import synth

REL_F32 = 1e-5        # relative L2 bound of the f32 CUDA-core paths
REL_TC = 5e-3         # relative L2 bound of the tensor-core path (16-bit operands, f32 accumulate)
W_ABS = 1e-6          # renormalised weights, absolute
# Router logits against the oracle's f64 logits, relative to the row's largest |logit|.
# rl_route forms each logit as one f32 dot product (at most a few hundred sequential terms
# per partial sum), which stays within 1e-6 of the row scale.
LOGIT_ROUTE = 1e-6
# moe_decode_stack adds its router partials across CTAs in 64-bit fixed point (2^-36 per CTA
# partial, then one f32 rounding of the sum and the RMSNorm scale applied to the summed dot),
# and its layer input is the GPU's own residual stream, which grows with depth; its bound is
# taken ten times wider.
LOGIT_FIXED = 1e-5


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def u64(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


class OracleSide:
    """Oracle inputs for a device model: routers, biases, residency rows and records, all
    from the generator; records looked up by the device slot addresses of the model."""

    def __init__(self, model):
        self.m = model
        self.w = model.w
        self.grid = synth.grid(self.w.seed)
        self._addr = model.expert_of_addr()
        self._cache = {}

    def record(self, slot: int) -> np.ndarray:
        le = self._addr[int(slot)]
        if le not in self._cache:
            self._cache[le] = synth.expert_records(self.w, le[0], le[1], 1)[0]
        return self._cache[le]

    def router(self, l):
        return synth.router(self.w, l)

    def bias(self, l):
        return synth.zipf_bias(self.w, l) if self.w.zipf_s > 0 else None

    def table_row(self, l):
        return self.m.table_host[l].copy()

    def experts(self, xn, ids, weights, slots):
        return oracle.moe_experts(xn, ids, weights, slots, self.record, self.w.hidden, self.w.inter, self.grid)


def check_route(gpu_logits, gpu_ids, gpu_w, gpu_slots, o_logits64, table_row, k, layer, report,
                logit_tol=LOGIT_ROUTE):
    """Decision protocol for the router.
    (i) the oracle's selection on the GPU's f32 logits equals the GPU's ids and slots
        bit-exactly, weights within W_ABS;
    (ii) the GPU's logits match the oracle's f64 logits within logit_tol of the row scale
        (LOGIT_ROUTE for rl_route, LOGIT_FIXED for the fused stack's fixed-point sums);
    (iii) the oracle's ids from its own logits equal the GPU's, except where two candidates
        are closer than the measured logit error (a genuine f32 near-tie), which is counted in
        report["near_ties"]; callers bound that count.  report["logit_err"] keeps the largest
        error seen, relative to the row scale."""
    r = oracle.route_from_logits(gpu_logits, table_row, k, layer)
    assert np.array_equal(r.ids, gpu_ids), "selection on the GPU's logits differs"
    assert np.array_equal(r.slots, gpu_slots), "slot lookup differs"
    assert np.max(np.abs(r.weights - gpu_w)) <= W_ABS, np.max(np.abs(r.weights - gpu_w))
    scale = np.max(np.abs(o_logits64), axis=1, keepdims=True)
    err = np.abs(gpu_logits.astype(np.float64) - o_logits64)
    rel = float(np.max(err / scale))
    report["logit_err"] = max(report.get("logit_err", 0.0), rel)
    assert rel <= logit_tol, (rel, logit_tol)
    own = oracle.select_topk(o_logits64.astype(np.float32), k)
    ties = 0
    for t in np.nonzero(np.any(own != gpu_ids, axis=1))[0]:
        # the two orders must differ only between candidates whose f64 gap is within the error
        eps = 4 * float(np.max(err[t])) + 1e-30
        a, b = own[t].tolist(), gpu_ids[t].tolist()
        lg = o_logits64[t]
        for i in range(k):
            if a[i] != b[i]:
                assert abs(lg[a[i]] - lg[b[i]]) <= eps, (t, a, b)
        ties += 1
    report["near_ties"] = report.get("near_ties", 0) + ties
    return r
