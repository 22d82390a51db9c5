"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small workloads are compared on every output; the full-size layer workloads
on the complete outputs of a sample of (window, KV head) groups, computed in
the same launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _check(inp, groups=None):
    gpu = gu.run_cuda(inp)
    ref = oracle.run(inp, groups=groups)
    err = gu.errors(gpu, ref, inp, groups)
    print(inp["workload"].name, err)
    gu.assert_within(err)
    return gpu


def test_tiny_workload():
    _check(synth.make_inputs(synth.workload("tiny")))


def test_qwen3_1p7b_layer_full():
    _check(synth.make_inputs(synth.workload("qwen3_1p7b")))


EDGE = [
    # hq, hkv, d, lp, lc
    dict(hq=2, hkv=1, head_dim=64, lp=[0], lc=[64]),          # no prefix: plain causal
    dict(hq=4, hkv=2, head_dim=128, lp=[300], lc=[1]),        # single chunk row
    dict(hq=4, hkv=4, head_dim=128, lp=[129], lc=[130]),      # g = 1, ragged tiles
    dict(hq=6, hkv=2, head_dim=64, lp=[257], lc=[77]),        # g = 3: 126-row tiles
    dict(hq=8, hkv=1, head_dim=128, lp=[1000], lc=[200]),     # g = 8
    dict(hq=4, hkv=2, head_dim=128, lp=[5, 0, 700, 128], lc=[37, 100, 0, 256]),  # varlen + empty
    dict(hq=2, hkv=2, head_dim=64, lp=[4096], lc=[3]),        # long prefix, many splits
    dict(hq=16, hkv=1, head_dim=128, lp=[700], lc=[50]),      # g = 16: 8-token tiles
    dict(hq=128, hkv=1, head_dim=64, lp=[200], lc=[5]),       # g = 128, the largest group
]


def _many_windows(n=600, seed=3):
    # more windows than the persistent kernels have threads, most of them
    # tiny and many empty: the schedule scan takes several windows per thread
    r = np.random.RandomState(seed)
    lp = r.randint(0, 49, size=n)
    lc = r.randint(0, 7, size=n)
    lp[::5] = 0
    lc[1::7] = 0
    lc[0] = 3
    return dict(hq=4, hkv=2, head_dim=64, lp=lp.tolist(), lc=lc.tolist())


EDGE.append(_many_windows())


@pytest.mark.parametrize("cfg", EDGE, ids=[str(i) for i in range(len(EDGE))])
def test_edge_shapes(cfg):
    w = synth.custom(**cfg, seed=11, dout_std=1.0)
    _check(synth.make_inputs(w))


def test_qwen3_8b_layer_sampled_groups():
    inp = synth.make_inputs(synth.workload("qwen3_8b"))
    _check(inp, groups=[(0, 0), (0, 5)])


def test_varlen8_sampled_groups():
    inp = synth.make_inputs(synth.workload("varlen8"))
    _check(inp, groups=[(2, 1), (3, 7), (5, 0)])


def test_deterministic_and_forward_independent_of_backward():
    inp = synth.make_inputs(synth.custom(hq=8, hkv=2, head_dim=128, lp=[2000, 300],
                                         lc=[200, 129], seed=3))
    a = gu.run_cuda(inp)
    b = gu.run_cuda(inp)
    c = gu.run_cuda(inp, backward=False)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(a["o"], c["o"]) and torch.equal(a["lse"], c["lse"])


def test_backward_workspace_contents_do_not_matter():
    """Everything the backward keeps in its workspace (the schedule's prefix
    arrays, the fp32 partials of the query tiles that CTA boundaries cut, the
    status word) is written in the call before it is read: a workspace full
    of arbitrary bytes, one reused by earlier calls and a fresh one give
    bitwise the same results."""
    import frozen_prefix_chunk_gb300 as cfa
    inp = synth.make_inputs(synth.custom(hq=8, hkv=2, head_dim=128, lp=[5000, 700, 0],
                                         lc=[200, 129, 64], seed=4))
    ref = gu.run_cuda(inp)
    d = gu.to_device(inp)
    args = gu.make_args(d)
    o, lse, _ = cfa.forward(args, d["q"])
    delta = cfa.backward_preprocess(args, o, d["dout"])
    n = cfa.workspace_size(args, cfa.WS_BACKWARD)
    g = torch.Generator(device="cuda").manual_seed(1)
    for fill in ("random", "ones", "reused", "reused"):
        if fill == "random":
            ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
        elif fill == "ones":
            ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
        dq, dk, dv, ws = cfa.backward(args, d["dout"], lse, delta, ws=ws)
        assert cfa.read_status(ws) == 0
        assert torch.equal(dq.cpu(), ref["dq"]), fill
        assert torch.equal(dk.cpu(), ref["dk"]) and torch.equal(dv.cpu(), ref["dv"]), fill


def test_dequant_q8_0_bit_exact():
    import frozen_prefix_chunk_gb300 as cfa
    x = torch.randn(4096, 128, generator=torch.Generator().manual_seed(9)) * 3
    blocks = synth.encode_q8_0(x)
    # also the corner codes the encoder never emits
    raw = blocks.clone().view(-1, 34)
    raw[0, 2] = 0x80       # code -128
    raw[1, 0:2] = torch.tensor([0x01, 0x00], dtype=torch.uint8)   # subnormal scale
    raw[2, 0:2] = torch.tensor([0x00, 0x80], dtype=torch.uint8)   # -0 scale
    blocks = raw.view_as(blocks)
    f32, bf = cfa.dequant_q8_0(blocks.cuda())
    rf64, rf32, rbf = oracle.dequant_q8_0(blocks.numpy())
    assert np.array_equal(f32.cpu().numpy().view(np.uint32), rf32.view(np.uint32))
    assert np.array_equal(bf.cpu().view(torch.int16).numpy().view(np.uint16), rbf)


Q8 = [
    dict(hq=4, hkv=2, head_dim=128, lp=[300, 0, 1000], lc=[77, 5, 256]),
    dict(hq=6, hkv=3, head_dim=64, lp=[513], lc=[130]),
]


@pytest.mark.parametrize("cfg", Q8, ids=[str(i) for i in range(len(Q8))])
def test_q8_0_prefix_edge_shapes(cfg):
    w = synth.custom(**cfg, prefix_dtype=synth.PREFIX_Q8_0, seed=5, dout_std=1.0)
    _check(synth.make_inputs(w))


def test_window_63k_q8_sampled_group():
    inp = synth.make_inputs(synth.workload("window_63k_q8"))
    _check(inp, groups=[(0, 3)])


def test_q8_0_prefix_equals_bf16_of_its_dequant_bitwise():
    # the q8_0 path multiplies with bf16(fp32(d) * q); feeding those bf16 values
    # as a bf16 prefix must give bitwise the same outputs
    w = synth.custom(hq=8, hkv=2, head_dim=128, lp=[700, 129], lc=[100, 256],
                     prefix_dtype=synth.PREFIX_Q8_0, seed=8)
    inp = synth.make_inputs(w)
    a = gu.run_cuda(inp)
    inp16 = dict(inp)
    for k in ("k_prefix", "v_prefix"):
        _, _, bf = oracle.dequant_q8_0(inp[k].numpy())
        inp16[k] = torch.from_numpy(bf.view(np.int16)).view(torch.bfloat16)
    inp16["workload"] = synth.custom(hq=8, hkv=2, head_dim=128, lp=[700, 129], lc=[100, 256],
                                     seed=8)
    b = gu.run_cuda(inp16)
    for k in a:
        assert torch.equal(a[k], b[k]), k


F16 = [
    dict(hq=8, hkv=2, head_dim=128, lp=[700, 0, 300], lc=[100, 5, 256]),
    dict(hq=6, hkv=3, head_dim=64, lp=[513], lc=[130]),
]


@pytest.mark.parametrize("cfg", F16, ids=[str(i) for i in range(len(F16))])
def test_f16_prefix_shapes(cfg):
    w = synth.custom(**cfg, prefix_dtype=synth.PREFIX_F16, seed=7, dout_std=1.0)
    _check(synth.make_inputs(w))


def test_f16_prefix_equals_bf16_of_its_values_bitwise():
    # the fp16 path multiplies with bf16(RNE(x)); feeding those bf16 values as
    # a bf16 prefix must give bitwise the same outputs
    cfg = dict(hq=8, hkv=2, head_dim=128, lp=[700, 129], lc=[100, 256])
    inp = synth.make_inputs(synth.custom(**cfg, prefix_dtype=synth.PREFIX_F16, seed=9))
    a = gu.run_cuda(inp)
    inp16 = dict(inp)
    for k in ("k_prefix", "v_prefix"):
        inp16[k] = inp[k].float().to(torch.bfloat16)
    inp16["workload"] = synth.custom(**cfg, seed=9)
    b = gu.run_cuda(inp16)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_quantize_q8_0_bit_exact():
    import frozen_prefix_chunk_gb300 as cfa
    g = torch.Generator().manual_seed(21)
    x = torch.randn(3000, 128, generator=g) * torch.rand(3000, 1, generator=g) * 20
    x[:3] = 0                                        # zero blocks
    x[3, :32] = 1e-38                                # tiny values
    x[4, :32] = 8323072.0                            # fp16 scale overflow
    x[5, :32] = torch.tensor([0.5, -0.5, 2.5, -2.5] * 8) * 2   # halves at d = 1/127 * 5
    xb = x.to(torch.bfloat16)
    got = cfa.quantize_q8_0(xb.cuda()).cpu().numpy()
    want = oracle.quantize_q8_0(_bf16_bits(xb))
    assert np.array_equal(got, want)


def test_quantize_q8_0_appends_into_a_cache_at_any_block():
    import frozen_prefix_chunk_gb300 as cfa
    x = (torch.randn(37, 64, generator=torch.Generator().manual_seed(22)) * 3).to(torch.bfloat16)
    cache = torch.full((100 * 34,), 0xAB, dtype=torch.uint8, device="cuda")
    start = 5 * 34                                   # 2-byte aligned, not 16-byte
    n = x.numel() // 32 * 34
    cfa.quantize_q8_0(x.cuda(), out=cache[start:start + n])
    c = cache.cpu().numpy()
    assert np.array_equal(c[start:start + n], oracle.quantize_q8_0(_bf16_bits(x)).reshape(-1))
    assert np.all(c[:start] == 0xAB) and np.all(c[start + n:] == 0xAB)


def _guarded(shape, dtype, fill, guard):
    """A tensor of `shape` with `guard` leading-dimension rows of `fill` on
    either side: (whole buffer, the inner view the library writes into)."""
    n = shape[0]
    full = torch.full((guard + n + guard,) + tuple(shape[1:]), fill, dtype=dtype, device="cuda")
    return full, full[guard:guard + n]


def test_outputs_have_no_stray_writes():
    # Every output and both workspaces sit between guard rows holding a
    # sentinel: a valid call (ragged and empty windows, split query blocks)
    # must leave every guard untouched and give the same bits as a call on
    # plain buffers.
    import frozen_prefix_chunk_gb300 as cfa
    w = synth.custom(hq=8, hkv=2, head_dim=128, lp=[2000, 0, 300, 4096], lc=[200, 64, 0, 129],
                     seed=12, dout_std=1.0)
    inp = synth.make_inputs(w)
    ref = gu.run_cuda(inp)
    d = gu.to_device(inp)
    args = gu.make_args(d)
    tc, G = sum(w.lc), 64
    bf, f32 = torch.bfloat16, torch.float32
    o_full, o = _guarded((tc, w.hq, w.head_dim), bf, -7.0, G)
    dq_full, dq = _guarded((tc, w.hq, w.head_dim), bf, -7.0, G)
    dk_full, dk = _guarded((tc, w.hkv, w.head_dim), bf, -7.0, G)
    dv_full, dv = _guarded((tc, w.hkv, w.head_dim), bf, -7.0, G)
    lse_full, lse = _guarded((w.hq * tc,), f32, -7.0, 1024)
    dl_full, dl = _guarded((w.hq * tc,), f32, -7.0, 1024)
    nf = cfa.workspace_size(args, cfa.WS_FORWARD)
    nb = cfa.workspace_size(args, cfa.WS_BACKWARD)
    wsf_full, wsf = _guarded((nf,), torch.uint8, 0xA5, 4096)
    wsb_full, wsb = _guarded((nb,), torch.uint8, 0xA5, 4096)
    lse, dl = lse.view(w.hq, tc), dl.view(w.hq, tc)
    cfa.forward(args, d["q"], o, lse, wsf)
    cfa.backward_preprocess(args, o, d["dout"], dl)
    cfa.backward(args, d["dout"], lse, dl, dq, dk, dv, wsb)
    assert cfa.read_status(wsf) == 0 and cfa.read_status(wsb) == 0
    torch.cuda.synchronize()
    for full, g in ((o_full, G), (dq_full, G), (dk_full, G), (dv_full, G), (lse_full, 1024),
                    (dl_full, 1024), (wsf_full, 4096), (wsb_full, 4096)):
        fill = 0xA5 if full.dtype == torch.uint8 else -7.0
        assert bool((full[:g] == fill).all()) and bool((full[-g:] == fill).all())
    got = dict(o=o, lse=lse, delta=dl, dq=dq, dk=dk, dv=dv)
    for k, v in got.items():
        assert torch.equal(v.cpu(), ref[k]), k
