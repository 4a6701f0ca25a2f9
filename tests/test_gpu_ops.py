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
