"""q3i8_op_attention_static (attention with library-owned scratch, no
allocation) against q3i8_op_attention with a caller workspace and against the
CPU oracle's attention, through the C ABI.  Kept in its own file, collected
last, so that it also runs after every other GPU test in the same process; it
passes alone as well."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 2e-5  # the attention tolerance of the op parity tests


@pytest.fixture(scope="module")
def pkg():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


def _case(lens, nh, nkv, hd, seed):
    import torch

    rng = np.random.default_rng(seed)
    cap = max(64, (max(lens) + 63) // 64 * 64)
    n = len(lens)
    dev = torch.device("cuda")
    bf = lambda shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16).view(
        torch.int16).to(dev)
    q = torch.from_numpy((rng.standard_normal((n, nh, hd)) * 2).astype(np.float32)).to(dev)
    return (q, bf((n, nkv, cap, hd)), bf((n, nkv, cap, hd)), torch.arange(n, dtype=torch.int32, device=dev),
            torch.tensor(lens, dtype=torch.int32, device=dev))


def _both(pkg, case, nkv, splits):
    import torch

    q, k, v, seq, ln = case
    ws = torch.empty(pkg.op_attention_workspace(q.shape[0], q.shape[1], q.shape[2], splits) // 4 + 4,
                     dtype=torch.float32, device=q.device)
    st = torch.zeros(2, dtype=torch.int32, device=q.device)
    ref = torch.full_like(q, float("nan"))
    got = torch.full_like(q, float("nan"))
    pkg.op_attention(q, k, v, seq, ln, nkv, splits, ref, ws, st[0:1])
    pkg.op_attention_static(q, k, v, seq, ln, nkv, splits, got, st[1:2])
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    return got.cpu().numpy(), ref.cpu().numpy()


def _vs_oracle(case, lens, got):
    q, k, v, _, _ = case
    qh = q.cpu().numpy()
    kh = k.cpu().numpy().view(np.uint16)
    vh = v.cpu().numpy().view(np.uint16)
    for r, L in enumerate(lens):
        np.testing.assert_allclose(got[r], oracle.attention(qh[r], kh[r], vh[r], L), rtol=RTOL, atol=ATOL)


# (lens, n_heads, n_kv_heads, head_dim, splits, seed)
CASES = [
    ([700, 129, 64, 1], 16, 8, 128, 8, 11),
    ([65, 300], 8, 2, 64, 3, 12),
    ([5, 64, 65, 200], 8, 8, 64, 4, 13),   # GQA group 1 (one query head per kv head)
    ([1, 33, 500], 16, 8, 128, 1, 14),     # one split: the merge takes a single state
]


def test_static_scratch_matches_workspace_and_oracle_twice_in_a_row(pkg):
    # calls back to back with different sizes and inputs: a call must not see
    # anything the one before left in the scratch
    for lens, nh, nkv, hd, splits, seed in CASES:
        case = _case(lens, nh, nkv, hd, seed)
        got, ref = _both(pkg, case, nkv, splits)
        assert np.isfinite(got).all()
        np.testing.assert_allclose(got, ref, rtol=RTOL, atol=ATOL)
        _vs_oracle(case, lens, got)


def test_static_scratch_at_its_limit(pkg):
    # 32 rows x 16 heads x 15 splits of 130 floats: 3,993,600 bytes of the
    # 4 MiB scratch; contexts long enough that every split has positions
    R, nh, nkv, hd, splits = 32, 16, 8, 128, 15
    need = pkg.op_attention_workspace(R, nh, hd, splits)
    assert pkg.OP_ATTENTION_STATIC_SCRATCH_BYTES - 266240 < need <= pkg.OP_ATTENTION_STATIC_SCRATCH_BYTES
    lens = [960 - 7 * r for r in range(R)]
    for seed in (21, 22):
        case = _case(lens, nh, nkv, hd, seed)
        got, ref = _both(pkg, case, nkv, splits)
        np.testing.assert_allclose(got, ref, rtol=RTOL, atol=ATOL)
        _vs_oracle(case, lens, got)


def test_static_scratch_rejects_sizes_beyond_limit(pkg):
    import torch

    R, nh, hd, splits = 32, 16, 128, 64
    assert pkg.op_attention_workspace(R, nh, hd, splits) > pkg.OP_ATTENTION_STATIC_SCRATCH_BYTES
    dev = torch.device("cuda")
    q = torch.zeros(R, nh, hd, device=dev)
    k = torch.zeros(R, 8, 64, hd, dtype=torch.int16, device=dev)
    with pytest.raises(pkg.Q3Error, match="static limit"):
        pkg.op_attention_static(q, k, k, torch.arange(R, dtype=torch.int32, device=dev),
                                torch.ones(R, dtype=torch.int32, device=dev), 8, splits, q)
