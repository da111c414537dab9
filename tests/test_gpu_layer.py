"""The evaluation layer on the GPU against the oracle: attention sublayer over
[SG(memory); current] with W_O and the post-norm feed-forward sublayer, then
a two-layer stream whose hidden-state memories advance with Tail_M.

Tolerance (the outputs are LayerNorm outputs, O(1)): max abs err <=
2^-5 max|ref| and mean abs err <= 2^-7 mean|ref|. Each output passes through
about six bf16 roundings of O(1) values (projections, attention output, the
two residual sums, the feed-forward hidden, the output), each <= 2^-8
relative, so an element can be off by ~6 * 2^-8 of the values it depends on;
the mean error measured is about 2^-8 mean|ref|. A wrong element or index
errs by O(|ref|), far above either bound."""
import numpy as np
import pytest

import oracle
import rxl_inputs as gen
from tests._harness import assert_no_device_error, ring_rows, to_dev, to_host

pytestmark = pytest.mark.gpu


def _rb(a):
    return gen.round_to(np.asarray(a, np.float64), "bf16")


def _weights(seed, H, d, dff, nrel):
    rng = np.random.default_rng(seed)
    r = lambda *s, std=1.0: _rb(rng.standard_normal(s) * std)
    dh = 64
    return dict(w_q=r(d, H * dh, std=d ** -0.5), w_k=r(d, H * dh, std=d ** -0.5),
                w_v=r(d, H * dh, std=d ** -0.5), w_o=r(H * dh, d, std=(H * dh) ** -0.5),
                r=_rb(gen.rel_table(nrel, 256, H, dh, seed, 9)), u=r(H, dh, std=0.02),
                vbias=r(H, dh, std=0.02), ln1_gamma=1 + r(d, std=0.1), ln1_beta=r(d, std=0.1),
                w_1=r(d, dff, std=d ** -0.5), b_1=r(dff, std=0.1), w_2=r(dff, d, std=dff ** -0.5),
                b_2=r(d, std=0.1), ln2_gamma=1 + r(d, std=0.1), ln2_beta=r(d, std=0.1))


def _check(name, got, ref):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert err.max() <= 2.0 ** -5 * np.abs(ref).max(), f"{name}: max err {err.max():.3e}"
    assert err.mean() <= 2.0 ** -7 * np.abs(ref).mean(), f"{name}: mean err {err.mean():.3e}"


class Layer:
    def __init__(self, w, B, H, L, cap, d, dff):
        import torch
        import long_context_lm_rel_gb300 as rxl
        self.rxl, self.torch = rxl, torch
        self.B, self.H, self.L, self.cap, self.d, self.dff = B, H, L, cap, d, dff
        self.dev = {k: to_dev(v, "bf16") for k, v in w.items()}
        self.W = rxl.make_layer_weights(**self.dev)

    def run(self, ring, m, head, h_in):
        rxl, torch = self.rxl, self.torch
        desc = rxl.make_desc(self.B, self.H, self.L, self.cap, m, head, 0.125)
        wsb = rxl.rxl_layer_fwd_workspace_bytes(desc, self.d, self.dff)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        out = torch.empty(self.B, self.L, self.d, device="cuda", dtype=torch.bfloat16)
        rxl.rxl_layer_fwd(desc, self.d, self.dff, self.W, ring, h_in, out, ws, wsb)
        return out


@pytest.mark.parametrize("B,H,L,cap,m,head,d,dff", [
    (2, 4, 150, 200, 180, 70, 256, 512),       # ragged tiles, wrapping ring, 2 column tiles
    (2, 16, 128, 256, 256, 0, 1024, 4096),     # model width of the benchmark configurations
    (1, 2, 64, 0, 0, 0, 256, 256),             # no memory
    (2, 8, 100, 130, 120, 20, 512, 320),       # W_O and W_1 split over 4 CTAs, W_1's last column tile 64 wide
    (2, 4, 512, 0, 0, 0, 256, 4096),           # W_1 in 256-wide blocks without a split, W_2 split with its LayerNorm
])
def test_layer_parity(B, H, L, cap, m, head, d, dff):
    import torch
    w = _weights(B + H + L, H, d, dff, cap + L)
    rng = np.random.default_rng(d)
    hm, hi = _rb(rng.standard_normal((B, m, d))), _rb(rng.standard_normal((B, L, d)))
    ring = np.zeros((B, max(cap, 1), d))
    if m:
        ring[:, ring_rows(cap, head, m)] = hm
    lay = Layer(w, B, H, L, cap, d, dff)
    out = lay.run(to_dev(ring, "bf16") if cap else None, m, head, to_dev(hi, "bf16"))
    torch.cuda.synchronize()
    assert_no_device_error()
    _check("h_out", to_host(out), oracle.layer_fwd(hm, hi, w, H, 0.125))


def test_two_layer_stream_with_hidden_state_memory():
    """Layers 0 and 1 over four segments; each layer's memory (its input
    states, Tail_M) lives in a ring advanced by rxl_mem_update. Every
    (segment, layer) output is checked against the oracle fed with the GPU's
    own layer input and memory contents, so the memory wiring is checked."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    B, H, L, cap, d, dff, layers, segments = 2, 4, 96, 160, 256, 512, 2, 4
    lays = [Layer(_weights(100 + n, H, d, dff, cap + L), B, H, L, cap, d, dff) for n in range(layers)]
    rings = [torch.zeros(B, cap, d, device="cuda", dtype=torch.bfloat16) for _ in range(layers)]
    state = [rxl.rxl_ring(rings[n].data_ptr(), B, cap, d, cap * d, rxl.RXL_DTYPE_BF16, 0, 0)
             for n in range(layers)]
    rng = np.random.default_rng(5)
    for seg in range(segments):
        h = to_dev(_rb(rng.standard_normal((B, L, d))), "bf16")
        for n in range(layers):
            st = state[n]
            m, head = st.len, st.head
            mem_logical = to_host(rings[n])[:, ring_rows(cap, head, m)] if m else np.zeros((B, 0, d))
            out = lays[n].run(rings[n], m, head, h)
            torch.cuda.synchronize()
            assert_no_device_error()
            ref = oracle.layer_fwd(mem_logical, to_host(h), {k: v for k, v in
                                   _weights(100 + n, H, d, dff, cap + L).items()}, H, 0.125)
            _check(f"segment {seg} layer {n}", to_host(out), ref)
            # Tail_M of the layer's input states, then the next layer's input
            rxl.rxl_mem_update(st, h, L * d, L)
            h = out
        torch.cuda.synchronize()
    assert state[0].len == min(cap, segments * L)
