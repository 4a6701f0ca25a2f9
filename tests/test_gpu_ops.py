"""Single-kernel parity through the C ABI's op entry points (GPU)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


def _bf16_bits(rng, shape, scale=1.0):
    import torch

    x = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def attention_case(pkg, lens, nh=16, nkv=8, hd=128, splits=8, seed=0):
    import torch

    rng = np.random.default_rng(seed)
    cap = max(64, (max(lens) + 63) // 64 * 64)
    n_seq = len(lens)
    k = _bf16_bits(rng, (n_seq, nkv, cap, hd))
    v = _bf16_bits(rng, (n_seq, nkv, cap, hd))
    q = (rng.standard_normal((n_seq, nh, hd)) * 2).astype(np.float32)
    dev = torch.device("cuda")
    tq = torch.from_numpy(q).to(dev)
    tk = torch.from_numpy(k.view(np.int16)).to(dev)
    tv = torch.from_numpy(v.view(np.int16)).to(dev)
    seq = torch.arange(n_seq, dtype=torch.int32, device=dev)
    ln = torch.tensor(lens, dtype=torch.int32, device=dev)
    out = torch.full((n_seq, nh, hd), float("nan"), device=dev)
    ws = torch.empty(pkg.op_attention_workspace(n_seq, nh, hd, splits) // 4 + 4, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkg.op_attention(tq, tk, tv, seq, ln, nkv, splits, out, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.cpu().numpy()
    for r, L in enumerate(lens):
        ref = oracle.attention(q[r], k[r], v[r], L)
        np.testing.assert_allclose(got[r], ref, rtol=1e-4, atol=2e-5)
    return got, (q, k, v)


@pytest.mark.parametrize("ctx", [1, 2, 63, 64, 65, 511, 512, 6144])
def test_attention_vs_oracle(pkg, ctx):
    attention_case(pkg, [ctx, max(1, ctx // 2), 1])


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_attention_split_count_invariant(pkg, splits):
    attention_case(pkg, [700, 129, 64], splits=splits, seed=splits)


def test_attention_head_dim_64_and_groups(pkg):
    attention_case(pkg, [100, 7], nh=4, nkv=2, hd=64, splits=2)
    attention_case(pkg, [300, 1], nh=8, nkv=1, hd=128, splits=4)


def test_attention_single_position_is_v(pkg):
    got, (q, k, v) = attention_case(pkg, [1, 1], nh=4, nkv=2, hd=64, splits=5)
    vv = (v.astype(np.uint32) << 16).view(np.float32)
    for r in range(2):
        for j in range(4):
            assert np.array_equal(got[r, j], vv[r, j // 2, 0])


def test_attention_rejects_bad_sizes(pkg):
    import torch

    dev = torch.device("cuda")
    q = torch.zeros(1, 4, 96, device=dev)
    k = torch.zeros(1, 2, 64, 96, dtype=torch.int16, device=dev)
    ws = torch.zeros(4096, device=dev)
    with pytest.raises(pkg.Q3Error):
        pkg.op_attention(q, k, k, torch.zeros(1, dtype=torch.int32, device=dev),
                         torch.ones(1, dtype=torch.int32, device=dev), 2, 1, q, ws)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (100, 256, 1024), (128, 128, 128), (300, 1024, 3072),
                                   (513, 384, 2048)])
def test_tc_gemm_vs_oracle(pkg, M, N, K):
    """The tcgen05 prefill projection against the oracle's int8 matmul on the value it multiplies (hi + lo,
    exact in fp32): several tiles, a ragged last row tile, a single row."""
    import torch

    rng = np.random.default_rng(M * 7 + N + K)
    x = (rng.standard_normal((M, K)) * 1.5).astype(np.float32)
    hi = x.astype(np.float16)
    lo = (x - hi.astype(np.float32)).astype(np.float16)
    xs = hi.astype(np.float32) + lo.astype(np.float32)
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    s = (rng.random(N) * 0.02 + 1e-3).astype(np.float32)
    ref = oracle.matmul_i8(q, s, xs, nthreads=oracle.default_threads())
    dev = torch.device("cuda")
    planes = torch.from_numpy(np.ascontiguousarray(np.concatenate([hi, lo], axis=1)).view(np.int16)).to(dev)
    y = torch.full((M, N), float("nan"), device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkg.op_gemm_i8(planes, torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev), y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = y.cpu().numpy()
    # two fp32 sums of the same K exact products in different orders (and the tensor core's own
    # accumulation): |err| <= 4 K eps32 sum|terms|; a layout or indexing error is O(sum|terms|)
    bound = 4 * K * 6e-8 * (s[None, :] * (np.abs(xs) @ np.abs(q.astype(np.float32)).T)) + 1e-6
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))


@pytest.mark.parametrize("M,N,K", [(256, 2048, 6144), (256, 4096, 2048), (130, 2048, 2048), (40, 1024, 1024)])
def test_tc_gemm_split_k_vs_oracle(pkg, M, N, K):
    """Short prompts on narrow projections (the 1.7B shape's O / down / QKV at 256 rows, a ragged row tile):
    K split over CTAs, partial sums added in split order by a second kernel.  Same bound as the unsplit GEMM,
    and the result equals itself run to run."""
    import torch

    ws_bytes = pkg.op_gemm_i8_splitk_workspace(M, N, K)
    assert ws_bytes > 0  # these shapes are split on a GB300 (152 SMs)
    rng = np.random.default_rng(M + N + K)
    x = (rng.standard_normal((M, K)) * 1.5).astype(np.float32)
    hi = x.astype(np.float16)
    lo = (x - hi.astype(np.float32)).astype(np.float16)
    xs = hi.astype(np.float32) + lo.astype(np.float32)
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    s = (rng.random(N) * 0.02 + 1e-3).astype(np.float32)
    ref = oracle.matmul_i8(q, s, xs, nthreads=oracle.default_threads())
    dev = torch.device("cuda")
    planes = torch.from_numpy(np.ascontiguousarray(np.concatenate([hi, lo], axis=1)).view(np.int16)).to(dev)
    dq, ds = torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = []
    for _ in range(2):
        y = torch.full((M, N), float("nan"), device=dev)
        pkg.op_gemm_i8_splitk(planes, dq, ds, y, ws, st)
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy())
    assert int(st.item()) == 0
    assert np.array_equal(outs[0], outs[1])
    bound = 4 * K * 6e-8 * (s[None, :] * (np.abs(xs) @ np.abs(q.astype(np.float32)).T)) + 1e-6
    assert np.all(np.abs(outs[0] - ref) <= bound), float(np.max(np.abs(outs[0] - ref) - bound))
    with pytest.raises(pkg.Q3Error, match="workspace"):
        pkg.op_gemm_i8_splitk(planes, dq, ds, torch.zeros(M, N, device=dev), ws[:16], st)


def test_tc_gemm_rejects_bad_shapes(pkg):
    import torch

    dev = torch.device("cuda")
    with pytest.raises(pkg.Q3Error):
        pkg.op_gemm_i8(torch.zeros(4, 192, dtype=torch.int16, device=dev), torch.zeros(100, 96, dtype=torch.int8,
                       device=dev), torch.ones(100, device=dev), torch.zeros(4, 100, device=dev))
