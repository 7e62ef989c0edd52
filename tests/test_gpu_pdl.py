"""Programmatic dependent launch: a decode chain whose kernels overlap must
give exactly the results of the same chain launched without PDL, eagerly and
under CUDA-graph capture, including the hazards PDL opens (a GEMV's output
read by the next producer; a q8 plane rewritten by the next step's producer
while the previous GEMV may still be reading it)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mq():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_quantized_gemv_gb300 import build
    build.build()
    import quant_quantized_gemv_gb300 as m
    m.lib()
    yield m
    m.mq_set_pdl(False)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class FfnChain:
    """rms -> gate, up (q4_K) -> swiglu -> down (q6_K): the FFN half of a
    14B-shaped layer at reduced width, all buffers preallocated."""

    def __init__(self, mq, hidden=2048, inter=5376, grouped=False):
        import torch
        self.grouped = grouped
        g = synth.rng("pdl-chain")
        self.mq, self.h, self.i = mq, hidden, inter
        self.Wg_h = synth.q4k_blocks(g, inter, hidden)
        self.Wu_h = synth.q4k_blocks(g, inter, hidden)
        self.Wd_h = synth.q6k_blocks(g, hidden, inter)
        self.Wg = dev(mq.mq_repack_q4k(self.Wg_h, inter, hidden))
        self.Wu = dev(mq.mq_repack_q4k(self.Wu_h, inter, hidden))
        self.Wd = dev(mq.mq_repack_q6k(self.Wd_h, hidden, inter))
        self.x = torch.empty(hidden, device="cuda")
        self.gain = dev(synth.normal(g, hidden, 1.0, 0.1))
        self.xn = torch.empty(hidden, device="cuda")
        self.q8a = torch.empty(mq.mq_q8_bytes(hidden), dtype=torch.uint8, device="cuda")
        self.yg = torch.empty(inter, device="cuda")
        self.yu = torch.empty(inter, device="cuda")
        self.act = torch.empty(inter, device="cuda")
        self.q8b = torch.empty(mq.mq_q8_bytes(inter), dtype=torch.uint8, device="cuda")
        self.out = torch.empty(hidden, device="cuda")
        self.wsg = mq.mq_gemv_workspace(inter, hidden)
        self.wsd = mq.mq_gemv_workspace(hidden, inter)
        self.wsgu = mq.mq_gemv_group_workspace([("q4k", self.Wg, inter), ("q4k", self.Wu, inter)],
                                               hidden)

    def step(self):
        mq = self.mq
        mq.mq_rmsnorm_quant_q8(self.x, self.gain, 1e-6, y=self.xn, q8=self.q8a)
        if self.grouped:                          # gate and up in one launch
            mq.mq_gemv_group_q8([("q4k", self.Wg, self.i), ("q4k", self.Wu, self.i)], self.q8a,
                                self.h, ys=[self.yg, self.yu], ws=self.wsgu)
        else:
            mq.mq_gemv_q4k_q8(self.Wg, self.q8a, self.i, self.h, y=self.yg, ws=self.wsg)
            mq.mq_gemv_q4k_q8(self.Wu, self.q8a, self.i, self.h, y=self.yu, ws=self.wsg)
        mq.mq_swiglu_quant_q8(self.yg, self.yu, y=self.act, q8=self.q8b)
        mq.mq_gemv_q6k_q8(self.Wd, self.q8b, self.h, self.i, y=self.out, ws=self.wsd)


def run_steps(mq, chain, xs, pdl, graph):
    import torch
    mq.mq_set_pdl(pdl)
    outs = []
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        if graph:
            chain.x.copy_(xs[0])
            chain.step()                          # warm-up outside capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                chain.step()
        for x in xs:
            chain.x.copy_(x)
            if graph:
                g.replay()
            else:
                chain.step()
            outs.append(chain.out.clone())
    torch.cuda.synchronize()
    mq.mq_set_pdl(False)
    return [o.cpu().numpy() for o in outs]


@pytest.mark.parametrize("grouped", [False, True])
def test_pdl_chain_is_bitwise_identical(mq, orc, grouped):
    chain = FfnChain(mq, grouped=grouped)
    g = synth.rng("pdl-inputs")
    xs = [dev(synth.normal(g, chain.h)) for _ in range(8)]
    ref = run_steps(mq, chain, xs, pdl=False, graph=False)
    for pdl, graph in ((True, False), (False, True), (True, True)):
        got = run_steps(mq, chain, xs, pdl=pdl, graph=graph)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b), (pdl, graph)
    # and every stage of the chain against the oracle, each fed what the
    # GPU's previous stage wrote (the buffers hold the last step, xs[-1],
    # identical in every run above): f32 producer outputs within 1e-4
    # relative, q8 planes bit-exact against the oracle's quantization of the
    # f32 values the producer wrote, GEMV outputs within 1e-4 * sum |terms|
    import torch
    torch.cuda.synchronize()
    hostv = lambda t: t.cpu().numpy()                        # noqa: E731
    x0 = xs[-1].cpu().numpy()
    xn = hostv(chain.xn)
    xn_ref = orc.rmsnorm(x0, chain.gain.cpu().numpy(), 1e-6)
    assert np.all(np.abs(xn - xn_ref) <= 1e-4 * np.abs(xn_ref) + 1e-30)
    d, q, s = orc.quantize_q8(xn)
    dg, qg, sg = mq.mq_q8_unpack_host(hostv(chain.q8a), chain.h)
    assert np.array_equal(d, dg) and np.array_equal(q, qg) and np.array_equal(s, sg)
    for W, yd in ((chain.Wg_h, chain.yg), (chain.Wu_h, chain.yu)):
        yref, absum = orc.gemv("q4k", W, d, q, chain.i, chain.h, threads=8)
        assert np.all(np.abs(hostv(yd).astype(np.float64) - yref) <= 1e-4 * absum)
    yg, yu = hostv(chain.yg), hostv(chain.yu)
    act = hostv(chain.act)
    act_ref = orc.swiglu(yg, yu)
    assert np.all(np.abs(act - act_ref) <= 1e-4 * np.abs(act_ref) + 1e-30)
    d2, q2, s2 = orc.quantize_q8(act)
    dg2, qg2, sg2 = mq.mq_q8_unpack_host(hostv(chain.q8b), chain.i)
    assert np.array_equal(d2, dg2) and np.array_equal(q2, qg2) and np.array_equal(s2, sg2)
    y, absum = orc.gemv("q6k", chain.Wd_h, d2, q2, chain.h, chain.i, threads=8)
    assert np.array_equal(hostv(chain.out), ref[-1])
    assert np.all(np.abs(ref[-1].astype(np.float64) - y) <= 1e-4 * absum)
