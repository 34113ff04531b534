"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Bar: packed codes, s_w, int8 activations and int32 accumulators bit-exact;
fp32 outputs within 1e-5 relative (the contract) -- the kernels perform the
same fp32 operations in the same order as the oracle, so the tests also
check that Y is bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle as O
import ternary_weight_linear_06_b300 as BL
from ternary_weight_linear_06_b300 import workloads as WL

pytestmark = pytest.mark.gpu

RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_y(Y_gpu, Y_ref):
    Y_gpu = np.asarray(Y_gpu, np.float32)
    Y_ref = np.asarray(Y_ref, np.float32)
    rel = np.abs(Y_gpu.astype(np.float64) - Y_ref) / np.maximum(np.abs(Y_ref.astype(np.float64)), 1e-30)
    assert rel.max(initial=0.0) <= RTOL, rel.max()
    np.testing.assert_array_equal(Y_gpu.view(np.uint32), Y_ref.view(np.uint32))


# ----------------------------------------------------------------- packing
def check_pack(W):
    packed, s_w = BL.pack(dev(W))
    p_ref, s_ref, t_ref = O.pack_weights(W)
    assert host(s_w).view(np.uint32)[0] == np.float32(s_ref).view(np.uint32), (host(s_w)[0], s_ref)
    np.testing.assert_array_equal(host(packed), p_ref)
    np.testing.assert_array_equal(host(BL.unpack(packed, W.shape[1])), t_ref)
    return packed, s_w, t_ref, s_ref


def test_pack_tiny():
    W, _ = WL.tiny_case(0)
    check_pack(W)


@pytest.mark.parametrize("shape", ["kv", "qo", "up", "down"])
def test_pack_decode_shapes(shape):
    check_pack(WL.decode_weights(shape, 0))


def test_pack_exponent_extremes_and_ties():
    rng = np.random.default_rng(21)
    W = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    # values outside the 128-bit window: subnormals, tiny normals, huge values
    W[0, :8] = np.array([1e-45, -2e-44, 3e-39, -1e-38, 1e-20, 3e15, -7e25, 2e30], np.float32)
    check_pack(W)
    # exact ternary ties: entries equal to +-s_w/2 for the matrix's own s_w
    W = (rng.standard_normal((128, 512)) * 0.02).astype(np.float32)
    for _ in range(3):
        s = O.pack_weights(W)[1]
        W[np.arange(0, 128, 2), 7] = np.float32(s) * np.float32(0.5)
        W[np.arange(1, 128, 2), 9] = -np.float32(s) * np.float32(0.5)
        W[5, 11] = np.nextafter(np.float32(s) * np.float32(0.5), np.float32(1))
    s = O.pack_weights(W)[1]
    assert O.tie_count(W, s) > 0
    check_pack(W)


def test_pack_nonfinite_gives_nan_scale():
    W = np.ones((4, 64), np.float32)
    W[1, 3] = np.inf
    _, s_w = BL.pack(dev(W))
    assert np.isnan(host(s_w)[0])


# ------------------------------------------------------------ quantization
def test_quant_act_f32_and_bf16():
    _, X = WL.tiny_case(0)
    q, m = BL.quant_act(dev(X))
    q_ref, m_ref = O.quant_act(X)
    np.testing.assert_array_equal(host(q), q_ref)
    np.testing.assert_array_equal(host(m).view(np.uint32), m_ref.view(np.uint32))
    xb = WL.batched_activations_bf16(16, 2560, seed=31)
    Xb = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    q, m = BL.quant_act(Xb)
    q_ref, m_ref = O.quant_act(O.bf16_bits_to_f32(xb))
    np.testing.assert_array_equal(host(q), q_ref)
    np.testing.assert_array_equal(host(m), m_ref)


def _tc_to_row_major(act, M, K):
    # fp16 slot s of a 16-column group holds column (s >> 1) + 8 * (s & 1)
    return act.astype(np.int32).reshape(M, K // 16, 8, 2).transpose(0, 1, 3, 2).reshape(M, K)


@pytest.mark.parametrize("M,K,dtype", [(296, 2560, "bf16"), (1000, 6912, "f32"), (3001, 2560, "f32"),
                                       (300, 16384, "f32"), (300, 65536, "bf16")])
def test_quant_act_many_rows(M, K, dtype):
    # From 2 rows per SM the rows stream through a shared-memory ring (4 slots
    # for rows up to 8 KB, 3 up to 16 KB, 2 up to 64 KB); longer rows keep one
    # CTA per row. Both layouts; the SubLN variant with a gain as well.
    if dtype == "bf16":
        xb = WL.batched_activations_bf16(M, K, seed=33 + M)
        Xd = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        X = O.bf16_bits_to_f32(xb)
    else:
        X = WL.prefill_activations(M, K, seed=34 + M)
        X[5] = 0.0
        Xd = dev(X)
    q_ref, m_ref = O.quant_act(X)
    q, m = BL.quant_act(Xd)
    np.testing.assert_array_equal(host(q), q_ref)
    np.testing.assert_array_equal(host(m).view(np.uint32), m_ref.view(np.uint32))
    act, m = BL.quant_act_tc(Xd)
    np.testing.assert_array_equal(_tc_to_row_major(host(act), M, K), q_ref)
    np.testing.assert_array_equal(host(m).view(np.uint32), m_ref.view(np.uint32))
    g = WL.norm_gain(K, seed=35 + M)
    q, m = BL.rmsnorm_quant(Xd, dev(g))
    q_ref, m_ref = O.rmsnorm_quant(X, g)
    np.testing.assert_array_equal(host(q), q_ref)
    assert_m_close(host(m), m_ref)


# ----------------------------------------------------------------- forward
def check_forward(W, X, x_is_bf16_bits=False):
    packed, s_w, t_ref, s_ref = check_pack(W)
    if x_is_bf16_bits:
        Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
        Xf = O.bf16_bits_to_f32(X)
    else:
        Xd, Xf = dev(X), X
    Y, acc = BL.forward(Xd, packed, s_w, return_acc=True)
    Y_ref, acc_ref, _, _ = O.forward(Xf, t_ref, s_ref)
    np.testing.assert_array_equal(host(acc), acc_ref)
    assert_y(host(Y), Y_ref)


def test_forward_tiny_case():
    W, X = WL.tiny_case(0)
    check_forward(W, X)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 16, 17])
def test_forward_token_counts_ragged_rows(M):
    # N = 203 rows is ragged for every row-group size; K = 320 spans several 16-byte chunks per lane pass
    W = WL.gaussian_weights(203, 320, 0.02, seed=40 + M, outlier_frac=0.01)
    X = WL.student_t(M, 320, seed=60 + M)
    X[0, :5] = 0.0
    check_forward(W, X)


@pytest.mark.parametrize("K", [64, 128, 2048, 2112, 4096])
def test_forward_k_sizes(K):
    W = WL.gaussian_weights(70, K, 0.02, seed=K)
    X = WL.student_t(3, K, seed=K + 1)
    check_forward(W, X)


def test_forward_bf16_input_batched():
    W = WL.decode_weights("kv", 3)
    xb = WL.batched_activations_bf16(4, 2560, seed=77)
    check_forward(W, xb, x_is_bf16_bits=True)


def test_forward_zero_and_extreme_tokens():
    W = WL.gaussian_weights(96, 256, 0.02, seed=5)
    X = np.zeros((4, 256), np.float32)
    X[1] = 1e-30                      # below eps: m = eps, q = 0
    X[2, 3] = 1e30                    # single huge entry
    X[3] = WL.student_t(1, 256, seed=6)[0] * np.float32(1e6)
    check_forward(W, X)


def test_forward_empty_is_noop():
    W = WL.gaussian_weights(32, 64, 0.02, seed=1)
    packed, s_w = BL.pack(dev(W))
    Y = BL.forward(torch.zeros((0, 64), device="cuda"), packed, s_w)
    assert Y.shape == (0, 32)


@pytest.mark.parametrize("shape", ["kv", "qo", "up", "down"])
def test_forward_decode_full_size_m1(shape):
    W = WL.decode_weights(shape, 1)
    X = WL.decode_activations(shape, 1)
    check_forward(W, X)


# --------------------------------------------------------------------- FFN
def test_ffn_small():
    D, F, M = 256, 512, 6
    Wu = WL.gaussian_weights(F, D, 0.02, seed=90, outlier_frac=0.001)
    Wd = WL.gaussian_weights(D, F, 0.02, seed=91, outlier_frac=0.001)
    X = WL.prefill_activations(M, D, seed=92)
    up, s_up = BL.pack(dev(Wu))
    down, s_down = BL.pack(dev(Wd))
    _, su, tu = O.pack_weights(Wu)
    _, sd, td = O.pack_weights(Wd)
    Y = BL.ffn(dev(X), up, s_up, down, s_down)
    Y_ref, _ = O.ffn(X, tu, su, td, sd)
    assert_y(host(Y), Y_ref)


def test_workspace_status_clean():
    assert BL.workspace_status() == 0


def test_forward_q8_shared_quantization():
    # q/k/v style: one quantization, three projections
    X = WL.decode_activations("qo", 2, M=3)
    q, m = BL.quant_act(dev(X))
    q_ref, m_ref = O.quant_act(X)
    np.testing.assert_array_equal(host(q), q_ref)
    for shape in ("qo", "kv"):
        W = WL.decode_weights(shape, 2)
        packed, s_w, t_ref, s_ref = check_pack(W)
        Y, acc = BL.forward_q8(q, m, packed, s_w, return_acc=True)
        acc_ref = O.int_matmul(q_ref, t_ref)
        np.testing.assert_array_equal(host(acc), acc_ref)
        assert_y(host(Y), O.dequant(acc_ref, s_ref, m_ref))
        Y2 = BL.forward(dev(X), packed, s_w)
        np.testing.assert_array_equal(host(Y2), host(Y))


# ------------------------------------------------------------------- batch
def _batch_case(specs, seed):
    """specs: list of (M, K, N, bf16, want_acc). Returns problems + oracle refs."""
    rng = np.random.default_rng(seed)
    probs, refs = [], []
    for i, (M, K, N, bf16, want_acc) in enumerate(specs):
        W = WL.gaussian_weights(N, K, 0.02, seed=seed * 100 + i, outlier_frac=0.001)
        packed, s_w, t_ref, s_ref = check_pack(W)
        if bf16:
            xb = WL.batched_activations_bf16(M, K, seed=seed * 100 + 50 + i)
            Xd = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
            Xf = O.bf16_bits_to_f32(xb)
        else:
            Xf = WL.student_t(M, K, seed=seed * 100 + 50 + i) * np.float32(rng.uniform(0.1, 10))
            Xd = dev(Xf)
        Y = torch.full((M, N), float("nan"), device="cuda")
        acc = torch.zeros((M, N), dtype=torch.int32, device="cuda") if want_acc else None
        probs.append((Xd, packed, s_w, Y, acc) if want_acc else (Xd, packed, s_w, Y))
        refs.append(O.forward(Xf, t_ref, s_ref))
    return probs, refs


def _check_batch(probs, refs):
    for prob, (Y_ref, acc_ref, _, _) in zip(probs, refs):
        assert_y(host(prob[3]), Y_ref)
        if len(prob) > 4:
            np.testing.assert_array_equal(host(prob[4]), acc_ref)


def test_forward_batch_mixed_problems():
    specs = [(1, 2560, 640, False, True), (1, 2560, 2560, False, False), (2, 320, 203, True, True),
             (3, 6912, 100, False, True), (5, 128, 64, False, True), (1, 64, 7, True, True),
             (4, 2048, 513, False, True), (0, 256, 16, False, False)]
    probs, refs = _batch_case(specs, seed=3)
    BL.forward_batch(probs)
    _check_batch(probs, refs)


def test_forward_batch_many_tiny_problems_next_to_a_large_one():
    # byte-balanced CTA runs put the tiny problems together; the launch plan
    # must split the batch when one run would touch too many problems
    specs = [(1, 4096, 2048, False, True)] + [(1, 64, 4, False, True)] * 60 + [(2, 128, 12, True, True)] * 20
    probs, refs = _batch_case(specs, seed=4)
    BL.forward_batch(probs)
    _check_batch(probs, refs)


def test_forward_batch_matches_single_calls_bitwise():
    specs = [(1, 2560, 640, False, True), (1, 6912, 256, False, True), (2, 2560, 96, False, True)]
    probs, _ = _batch_case(specs, seed=5)
    BL.forward_batch(probs)
    for X, packed, s_w, Y, acc in probs:
        Y1, acc1 = BL.forward(X, packed, s_w, return_acc=True)
        np.testing.assert_array_equal(host(Y1).view(np.uint32), host(Y).view(np.uint32))
        np.testing.assert_array_equal(host(acc1), host(acc))


def test_forward_batch_prequantized_inputs():
    # BL_DTYPE_I8 problems (int8 + per-token scales) next to fp32 and bf16 ones
    specs = [(1, 2560, 640, False, True), (3, 6912, 256, True, True), (2, 2560, 96, False, True)]
    probs, refs = _batch_case(specs, seed=7)
    mixed = []
    for i, (X, packed, s_w, Y, acc) in enumerate(probs):
        if i != 1:
            q, m = BL.quant_act(X)
            mixed.append((q, packed, s_w, Y, acc, m))
        else:
            mixed.append((X, packed, s_w, Y, acc))
    BL.forward_batch(mixed)
    _check_batch(probs, refs)


def test_forward_long_k_and_tiny_n():
    for (M, K, N) in [(1, 65536, 8), (3, 65536, 5), (2, 16384, 4), (1, 28672, 130)]:
        W = WL.gaussian_weights(N, K, 0.01, seed=K + N)
        X = WL.student_t(M, K, seed=K + N + 1)
        check_forward(W, X)


# ------------------------------------------------- tensor-core GEMM (M >= 5)
@pytest.mark.parametrize("M,K,N", [(17, 64, 128), (64, 320, 203), (128, 2560, 640), (129, 576, 130),
                                   (300, 2560, 257), (1000, 128, 384)])
def test_gemm_path_ragged_tiles(M, K, N):
    # several 128-token and 128-row tiles with ragged tails, K from one to 40 steps
    W = WL.gaussian_weights(N, K, 0.02, seed=M + K + N, outlier_frac=0.001)
    X = WL.prefill_activations(M, K, seed=M * 7 + K)
    X[min(3, M - 1)] = 0.0
    check_forward(W, X)


def test_gemm_path_bf16_batched_decode_inputs():
    W = WL.decode_weights("up", 0)
    xb = WL.batched_activations_bf16(64, 2560, seed=78)
    check_forward(W, xb, x_is_bf16_bits=True)


def test_gemm_exact_at_the_accumulator_bound():
    # every q = 127 and every t = +1 at K = 65536: acc = 127 * 65536 = 8,323,072 (< 2^24)
    M, K, N = 20, 65536, 16
    W = np.full((N, K), 0.5, np.float32)
    W[1::2] = -0.5                                     # alternate rows all -1
    X = np.ones((M, K), np.float32)
    X[1] = -1.0
    packed, s_w, t_ref, s_ref = check_pack(W)
    Y, acc = BL.forward(dev(X), packed, s_w, return_acc=True)
    Y_ref, acc_ref, _, _ = O.forward(X, t_ref, s_ref)
    assert acc_ref[0, 0] == 127 * K and acc_ref[0, 1] == -127 * K
    np.testing.assert_array_equal(host(acc), acc_ref)
    assert_y(host(Y), Y_ref)


def test_gemm_exact_large_plus_small_partial_sums():
    # a large running sum followed by many +-1 contributions: truncating
    # accumulation would lose the small terms
    M, K, N = 32, 16384, 64
    rng = np.random.default_rng(5)
    X = np.empty((M, K), np.float32)
    X[:, : K // 2] = 127.0                             # q = 127 on the first half
    X[:, K // 2:] = rng.choice([-1.0, 1.0], size=(M, K // 2)).astype(np.float32)   # q = +-1 after scaling
    W = rng.choice([-0.5, 0.0, 0.5], size=(N, K)).astype(np.float32)
    W[:, : K // 2] = 0.5
    check_forward(W, X)


def test_gemm_ffn_prefill_block():
    D, F, M = 256, 640, 200
    Wu = WL.gaussian_weights(F, D, 0.02, seed=93, outlier_frac=0.001)
    Wd = WL.gaussian_weights(D, F, 0.02, seed=94, outlier_frac=0.001)
    X = WL.prefill_activations(M, D, seed=95)
    up, s_up = BL.pack(dev(Wu))
    down, s_down = BL.pack(dev(Wd))
    _, su, tu = O.pack_weights(Wu)
    _, sd, td = O.pack_weights(Wd)
    Y = BL.ffn(dev(X), up, s_up, down, s_down)
    Y_ref, _ = O.ffn(X, tu, su, td, sd)
    assert_y(host(Y), Y_ref)


def test_gemm_forward_q8_prequantized():
    M, K, N = 96, 2560, 640
    X = WL.prefill_activations(M, K, seed=97)
    W = WL.decode_weights("kv", 4)
    q, m = BL.quant_act(dev(X))
    packed, s_w, t_ref, s_ref = check_pack(W)
    Y, acc = BL.forward_q8(q, m, packed, s_w, return_acc=True)
    q_ref, m_ref = O.quant_act(X)
    acc_ref = O.int_matmul(q_ref, t_ref)
    np.testing.assert_array_equal(host(acc), acc_ref)
    assert_y(host(Y), O.dequant(acc_ref, s_ref, m_ref))


def test_gemm_and_gemv_agree_bitwise_across_the_switch():
    # the same token rows through the GEMV (4 tokens) and the GEMM (all tokens)
    W = WL.decode_weights("qo", 6)
    X = WL.student_t(40, 2560, seed=98)
    packed, s_w = BL.pack(dev(W))
    Y_all, acc_all = BL.forward(dev(X), packed, s_w, return_acc=True)
    Y_few, acc_few = BL.forward(dev(X[:4]), packed, s_w, return_acc=True)
    np.testing.assert_array_equal(host(acc_all)[:4], host(acc_few))
    np.testing.assert_array_equal(host(Y_all)[:4].view(np.uint32), host(Y_few).view(np.uint32))
    assert BL.workspace_status() == 0


def test_forward_tc_matches_the_oracle_and_forward():
    # the tensor-core operand form: quantize once, run the contraction only
    for M, K, N in [(5, 2560, 640), (256, 6912, 257)]:
        W = WL.gaussian_weights(N, K, 0.02, seed=K + N + M, outlier_frac=0.001)
        X = WL.prefill_activations(M, K, seed=M + 99)
        packed, s_w, t_ref, s_ref = check_pack(W)
        act, m = BL.quant_act_tc(dev(X))
        Y, acc = BL.forward_tc(act, m, packed, s_w, return_acc=True)
        Y_ref, acc_ref, q_ref, m_ref = O.forward(X, t_ref, s_ref)
        np.testing.assert_array_equal(host(act).astype(np.int32).reshape(M, K // 16, 8, 2).transpose(0, 1, 3, 2)
                                      .reshape(M, K), q_ref)
        np.testing.assert_array_equal(host(m).view(np.uint32), m_ref.view(np.uint32))
        np.testing.assert_array_equal(host(acc), acc_ref)
        assert_y(host(Y), Y_ref)
        Y2 = BL.forward(dev(X), packed, s_w)
        np.testing.assert_array_equal(host(Y2).view(np.uint32), host(Y).view(np.uint32))


# full-size prefill shapes: every tile shape of the GEMM (the host picks 256-,
# 192- or 128-token tiles from the tile count), checked on sampled token rows
def _sampled_rows(M, seed):
    rng = np.random.default_rng(seed)
    rows = {0, 1, M - 1, M - 2, M // 2}
    for tile in (128, 192, 256):
        rows.update(r for r in (tile - 1, tile, 3 * tile - 1, 3 * tile) if r < M)
    rows.update(rng.choice(M, size=min(24, M), replace=False).tolist())
    return np.array(sorted(rows))


def _check_sampled(W, X, seed):
    M = X.shape[0]
    packed, s_w = BL.pack(dev(W))
    _, s_ref, t_ref = O.pack_weights(W)
    Y, acc = BL.forward(dev(X), packed, s_w, return_acc=True)
    rows = _sampled_rows(M, seed)
    q_ref, m_ref = O.quant_act(X[rows])
    acc_ref = (q_ref.astype(np.float64) @ t_ref.astype(np.float64).T).astype(np.int64)   # exact: |acc| < 2^53
    np.testing.assert_array_equal(host(acc)[rows], acc_ref)
    assert_y(host(Y)[rows], O.dequant(acc_ref, s_ref, m_ref))


@pytest.mark.parametrize("shape", ["qo", "kv", "up", "down"])
def test_gemm_full_size_prefill_sampled_rows(shape):
    K, N = WL.SHAPES_2B[shape]
    _check_sampled(WL.decode_weights(shape, 3), WL.prefill_activations(4096, K, seed=300 + K + N), 17)


@pytest.mark.parametrize("M", [512, 2048])
def test_gemm_70b_class_shape_sampled_rows(M):
    K, N = 8192, 8192
    _check_sampled(WL.gaussian_weights(N, K, 0.01, seed=M, outlier_frac=0.001), WL.student_t(M, K, seed=M + 1), 19)


def test_gemm_split_k_ffn_few_tokens():
    # 16 tokens: the GEMM cuts K into parts (exact integer partial sums added
    # in the workspace), then ReLU^2 and the requantization run on the sums
    D, F, M = 2560, 6912, 16
    Wu = WL.decode_weights("up", 5)
    Wd = WL.decode_weights("down", 5)
    X = WL.student_t(M, D, seed=96)
    up, s_up = BL.pack(dev(Wu))
    down, s_down = BL.pack(dev(Wd))
    _, su, tu = O.pack_weights(Wu)
    _, sd, td = O.pack_weights(Wd)
    Y = BL.ffn(dev(X), up, s_up, down, s_down)
    Y_ref, _ = O.ffn(X, tu, su, td, sd)
    assert_y(host(Y), Y_ref)
    assert BL.workspace_status() == 0


@pytest.mark.parametrize("M", [9, 12, 33, 128])
def test_gemm_split_k_token_counts(M):
    for shape in ("qo", "kv", "down"):
        K, N = WL.SHAPES_2B[shape]
        W = WL.decode_weights(shape, 8)
        xb = WL.batched_activations_bf16(M, K, seed=800 + M)
        check_forward(W, xb, x_is_bf16_bits=True)


@pytest.mark.parametrize("shape,M", [("up", 64), ("down", 512), ("down", 9)])
def test_large_ffn_shapes_sampled_rows(shape, M):
    # 70B-class FFN shapes (K or N = 28672): the GEMM with split-K (64 and 9
    # tokens) and with 128/192/256-token tiles (512 tokens)
    K, N = WL.SHAPES_70B[shape]
    _check_sampled(WL.large_weights(shape), WL.student_t(M, K, seed=M + K), 23)


# -------------------------------------------------------------- gated FFN
@pytest.mark.parametrize("M", [1, 4, 16, 200])
def test_gated_ffn_all_paths(M):
    # 1 and 4 tokens: GEMV; 16: split-K GEMM; 200: tiled GEMM
    D, F = 256, 640
    Wu = WL.gaussian_weights(F, D, 0.02, seed=110 + M, outlier_frac=0.001)
    Wg = WL.gaussian_weights(F, D, 0.02, seed=120 + M, outlier_frac=0.001)
    Wd = WL.gaussian_weights(D, F, 0.02, seed=130 + M, outlier_frac=0.001)
    X = WL.prefill_activations(M, D, seed=140 + M)
    up, s_up = BL.pack(dev(Wu))
    gate, s_gate = BL.pack(dev(Wg))
    down, s_down = BL.pack(dev(Wd))
    _, su, tu = O.pack_weights(Wu)
    _, sg, tg = O.pack_weights(Wg)
    _, sd, td = O.pack_weights(Wd)
    Y = BL.ffn_gated(dev(X), up, s_up, gate, s_gate, down, s_down)
    Y_ref, _ = O.ffn_gated(X, tu, su, tg, sg, td, sd)
    assert_y(host(Y), Y_ref)
    assert BL.workspace_status() == 0


def test_gated_ffn_2b_shapes_split_k():
    D, F, M = 2560, 6912, 12
    Wu, Wg, Wd = WL.decode_weights("up", 6), WL.decode_weights("up", 7), WL.decode_weights("down", 6)
    X = WL.student_t(M, D, seed=150)
    up, s_up = BL.pack(dev(Wu))
    gate, s_gate = BL.pack(dev(Wg))
    down, s_down = BL.pack(dev(Wd))
    _, su, tu = O.pack_weights(Wu)
    _, sg, tg = O.pack_weights(Wg)
    _, sd, td = O.pack_weights(Wd)
    Y = BL.ffn_gated(dev(X), up, s_up, gate, s_gate, down, s_down)
    Y_ref, _ = O.ffn_gated(X, tu, su, tg, sg, td, sd)
    assert_y(host(Y), Y_ref)


# ----------------------------------------------------------------- SubLN RMSNorm fused into the quantization
# Codes and accumulators are bit-exact. The norm factor comes from a
# compensated fp32 sum of squares on the GPU and from the exact sum in the
# oracle, so a token scale m may sit one fp32 step off where the exact value
# is that close to a rounding boundary; where m agrees, Y agrees bit for bit.
def assert_m_close(m_gpu, m_ref):
    a = np.asarray(m_gpu, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(m_ref, np.float32).view(np.int32).astype(np.int64)
    assert np.all(a > 0) and np.all(b > 0)
    d = np.abs(a - b)
    assert d.max(initial=0) <= 1, d.max()
    return d == 0


def assert_y_norm(Y_gpu, Y_ref, m_same):
    Y_gpu = np.asarray(Y_gpu, np.float32)
    Y_ref = np.asarray(Y_ref, np.float32)
    rel = np.abs(Y_gpu.astype(np.float64) - Y_ref) / np.maximum(np.abs(Y_ref.astype(np.float64)), 1e-30)
    assert rel.max(initial=0.0) <= RTOL, rel.max()
    np.testing.assert_array_equal(Y_gpu[m_same].view(np.uint32), Y_ref[m_same].view(np.uint32))


def _norm_rows(M, K, seed, dtype):
    X = WL.prefill_activations(M, K, seed=seed)
    if M >= 4:
        X[1] = 0.0                                   # all-zero token: codes 0, scale eps * r
        X[2] *= np.float32(1e-20)                    # far below eps_norm
        X[3] = np.float32(-3.5)                      # constant token
    if M >= 5:
        X[4] *= np.float32(1e15)                     # sum of squares near 1e34, still finite in fp32
    if dtype == "bf16":
        bits = WL.f32_to_bf16_bits(X)
        return bits, O.bf16_bits_to_f32(bits)
    return X, X


@pytest.mark.parametrize("M,K,dtype,gain", [
    (1, 2560, "f32", True), (3, 64, "bf16", False), (6, 6912, "f32", True), (64, 2560, "bf16", True),
    (257, 320, "f32", True), (2, 65536, "f32", True), (5, 65536, "bf16", False)])
def test_rmsnorm_quant_matches_oracle(M, K, dtype, gain):
    X_in, X32 = _norm_rows(M, K, 300 + M, dtype)
    g = WL.norm_gain(K, seed=310 + M) if gain else None
    Xd = dev(X_in).view(torch.bfloat16) if dtype == "bf16" else dev(X_in)
    q, m = BL.rmsnorm_quant(Xd, None if g is None else dev(g))
    q_ref, m_ref = O.rmsnorm_quant(X32, g)
    np.testing.assert_array_equal(host(q), q_ref)
    assert_m_close(host(m), m_ref)


@pytest.mark.parametrize("M,N,K", [(1, 2560, 2560), (4, 640, 2560), (9, 6912, 2560), (16, 2560, 6912),
                                   (200, 1000, 320), (1000, 384, 512)])
def test_forward_rmsnorm_all_paths(M, N, K):
    # 1 and 4 tokens: GEMV; 9 and 16: split-K GEMM; 200 and 1000: tiled GEMM
    W = WL.gaussian_weights(N, K, 0.02, seed=320 + M, outlier_frac=0.001)
    X, _ = _norm_rows(M, K, 330 + M, "f32")
    g = WL.norm_gain(K, seed=340 + M)
    packed, s_w = BL.pack(dev(W))
    _, s_ref, t_ref = O.pack_weights(W)
    Y, acc = BL.forward_rmsnorm(dev(X), packed, s_w, dev(g), return_acc=True)
    Y_ref, acc_ref, _, m_ref = O.forward_rmsnorm(X, t_ref, s_ref, g)
    np.testing.assert_array_equal(host(acc), acc_ref)
    _, m = BL.rmsnorm_quant(dev(X), dev(g))
    same = assert_m_close(host(m), m_ref)
    assert_y_norm(host(Y), Y_ref, same)
    assert BL.workspace_status() == 0


def test_rmsnorm_quant_feeds_the_decode_batch():
    # one norm + quantization of a token, shared by q, k and v as prequantized
    # batch problems, equals three forwards on RMSNorm(x)
    K = 2560
    X = WL.decode_activations("qo", 0, M=2)
    g = WL.norm_gain(K, seed=350)
    q, m = BL.rmsnorm_quant(dev(X), dev(g))
    probs, refs = [], []
    for i, shape in enumerate(("qo", "kv", "kv")):
        W = WL.decode_weights(shape, 40 + i)
        packed, s_w = BL.pack(dev(W))
        _, s_ref, t_ref = O.pack_weights(W)
        Y = torch.empty((2, W.shape[0]), dtype=torch.float32, device="cuda")
        probs.append((q, packed, s_w, Y, None, m))
        refs.append(O.forward_rmsnorm(X, t_ref, s_ref, g))
    BL.forward_batch(probs)
    _, m_ref = O.rmsnorm_quant(X, g)
    same = assert_m_close(host(m), m_ref)
    for (_, _, _, Y, _, _), (Y_ref, _, _, _) in zip(probs, refs):
        assert_y_norm(host(Y), Y_ref, same)


def _check_ffn_subln(Y_gpu, X, tu, su, td, sd, g_in, g_sub, tg=None, sg=None):
    # The GPU's h equals the oracle's wherever the input scale m agrees; a
    # scale one fp32 step off moves h by about one step, which can flip a code
    # of h only where 127 u / m lies within 1e-4 of a half-integer. Each such
    # code may move Y by one dequant step times |t|; nothing else may differ.
    Y_ref, h = O.ffn_subln(X, tu, su, td, sd, g_in=g_in, g_sub=g_sub, t_gate=tg, s_gate=sg)
    u = h if g_sub is None else (h * g_sub[None, :]).astype(np.float32)
    m_u = np.maximum(np.abs(u).max(axis=1), O.EPS).astype(np.float32)
    v = (u * np.float32(127)) / m_u[:, None]
    amb = np.abs(np.abs(v - np.floor(v)) - 0.5) < 1e-4
    _, m_h = O.rmsnorm_quant(h, g_sub)
    step = float(sd) * m_h.astype(np.float64) / 127.0
    slack = step[:, None] * (amb.astype(np.float64) @ np.abs(td.astype(np.float64)).T)
    Y_gpu = np.asarray(Y_gpu, np.float32).astype(np.float64)
    err = np.abs(Y_gpu - Y_ref.astype(np.float64))
    assert np.all(err <= RTOL * np.abs(Y_ref.astype(np.float64)) + 1.001 * slack), (err.max(), int(amb.sum()))


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("M", [1, 4, 16, 200])
def test_ffn_subln_all_paths(M, gated):
    D, F = 256, 640
    Wu = WL.gaussian_weights(F, D, 0.02, seed=360 + M, outlier_frac=0.001)
    Wg = WL.gaussian_weights(F, D, 0.02, seed=370 + M, outlier_frac=0.001)
    Wd = WL.gaussian_weights(D, F, 0.02, seed=380 + M, outlier_frac=0.001)
    X = WL.prefill_activations(M, D, seed=390 + M)
    g_in, g_sub = WL.norm_gain(D, seed=400 + M), WL.norm_gain(F, seed=410 + M)
    up, s_up = BL.pack(dev(Wu))
    gate, s_gate = BL.pack(dev(Wg))
    down, s_down = BL.pack(dev(Wd))
    _, su, tu = O.pack_weights(Wu)
    _, sg, tg = O.pack_weights(Wg)
    _, sd, td = O.pack_weights(Wd)
    kw = dict(gate=gate, s_gate=s_gate) if gated else {}
    Y = BL.ffn_subln(dev(X), up, s_up, down, s_down, g_in=dev(g_in), g_sub=dev(g_sub), **kw)
    _check_ffn_subln(host(Y), X, tu, su, td, sd, g_in, g_sub, *((tg, sg) if gated else ()))
    assert BL.workspace_status() == 0


@pytest.mark.parametrize("M", [1, 12])
def test_ffn_subln_2b_shapes_unit_gains(M):
    D, F = 2560, 6912
    Wu, Wg, Wd = WL.decode_weights("up", 8), WL.decode_weights("up", 9), WL.decode_weights("down", 8)
    X = WL.student_t(M, D, seed=420 + M)
    up, s_up = BL.pack(dev(Wu))
    gate, s_gate = BL.pack(dev(Wg))
    down, s_down = BL.pack(dev(Wd))
    _, su, tu = O.pack_weights(Wu)
    _, sg, tg = O.pack_weights(Wg)
    _, sd, td = O.pack_weights(Wd)
    Y = BL.ffn_subln(dev(X), up, s_up, down, s_down, gate=gate, s_gate=s_gate)
    _check_ffn_subln(host(Y), X, tu, su, td, sd, None, None, tg, sg)
