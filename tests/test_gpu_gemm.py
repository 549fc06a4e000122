"""GPU parity of the fused W8A8 GEMM against the oracle.

int32 accumulators must be bit-identical (also against torch._int_mm, the
pages' own check); bf16 outputs must be within one bf16 ulp (|d| <= 2^-7|y| +
1e-6), cosine >= 0.99999, no NaN/Inf.  Shapes span several tiles, ragged M/N/K
tails, the split-K path and adversarial +-127 operands that would overflow
fp32 exactness without the chunked accumulation.  The full-size DiT layers
are compared element by element in test_gpu_full_parity.py."""
import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import inputs
from tests._util import assert_bf16_exact, gpu_bf16_bits, to_dev

pytestmark = pytest.mark.gpu

SKINNY_DEFAULT = 16    # the library's default weight-streaming threshold

INT_SHAPES = [
    (64, 128, 256),
    (1, 8, 16),
    (7, 24, 48),
    (129, 136, 272),
    (256, 384, 1024),
    (300, 200, 1040),
    (2, 9216, 3072),       # skinny: split-K
    (16, 3072, 12288),     # few tokens, deep: cluster split-K
    (32, 3072, 12288),     # tiled, split-K
    (1024, 1024, 4096),
]


@pytest.mark.parametrize("M,N,K", INT_SHAPES)
def test_gemm_int32_matches_oracle(orc, M, N, K):
    a = inputs.random_int8(M, K, seed=M + K)
    w = inputs.random_int8(N, K, seed=N + 3 * K)
    c = i8.gemm_int32(to_dev(a), to_dev(w))
    i8.sync_check()
    got = c.cpu().numpy()
    want = orc.gemm_s32(a.numpy(), w.numpy())
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("M,N,K", [(64, 128, 256), (256, 384, 1024), (1024, 1024, 4096)])
def test_gemm_int32_matches_torch_int_mm(M, N, K):
    a = to_dev(inputs.random_int8(M, K, seed=5 + M))
    w = to_dev(inputs.random_int8(N, K, seed=6 + N))
    c = i8.gemm_int32(a, w)
    ref = torch._int_mm(a, w.t())
    assert torch.equal(c, ref)


def _adversarial(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.full((M, K), 127, dtype=torch.int8)
    w = torch.full((N, K), 127, dtype=torch.int8)
    # rows 1..: random signs at full magnitude; row 2: large then small terms
    sa = torch.randint(0, 2, (M, K), generator=g, dtype=torch.int8) * 2 - 1
    sw = torch.randint(0, 2, (N, K), generator=g, dtype=torch.int8) * 2 - 1
    a[1:] *= sa[1:]
    w[1:] *= sw[1:]
    if M > 2:
        a[2, K // 2:] = 1
    if N > 2:
        w[2, K // 2:] = -1
    a[min(3, M - 1)] = -127
    return a, w


@pytest.mark.parametrize("chunk_k", [64, 256, 512, 1024])
@pytest.mark.parametrize("M,N,pair", [(130, 136, 1), (260, 264, 2)], ids=["single_cta", "cta_pair"])
def test_gemm_int32_adversarial_exact(orc, chunk_k, M, N, pair):
    """+-127 operands: partial sums reach 127^2 * chunk_k; K = 8192 overflows
    fp32 exactness (2^24) unless the accumulation is chunked correctly."""
    K = 8192
    a, w = _adversarial(M, N, K, seed=chunk_k)
    i8.set_option("chunk_k", chunk_k)
    i8.set_option("cta_pair", pair)
    try:
        c = i8.gemm_int32(to_dev(a), to_dev(w))
        i8.sync_check()
    finally:
        i8.set_option("chunk_k", 1024)
        i8.set_option("cta_pair", 0)
    got = c.cpu().numpy()
    want = orc.gemm_s32(a.numpy(), w.numpy())
    assert got[0, 0] == 127 * 127 * K
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"chunk {chunk_k}: {len(bad)} mismatches, first {bad[:4].tolist()}"


def test_gemm_int32_extreme_k():
    """K = 131072 (the int32 bound): +127 x +127 gives 2114060288 exactly."""
    M, N, K = 2, 16, 131072
    a = torch.full((M, K), 127, dtype=torch.int8, device="cuda")
    w = torch.full((N, K), 127, dtype=torch.int8, device="cuda")
    w[1] = -127
    c = i8.gemm_int32(a, w)
    i8.sync_check()
    assert int(c[0, 0]) == 2114060288
    assert int(c[1, 1]) == -2114060288


def _oracle_linear_rows(orc, x, w, b, rows):
    """Oracle y for the selected rows (per-token quant is row-local)."""
    xs = inputs.bits(x[rows])
    aq, s_a = orc.quant_rows(xs)
    wq, s_w = orc.quant_rows(inputs.bits(w))
    acc = orc.gemm_s32(aq, wq)
    return orc.dequant_bias(acc, s_a, s_w, None if b is None else inputs.bits(b))


def _gpu_linear(x, w, b, widened=False):
    wq, s_w = i8.quant_weight_perchannel(to_dev(w))
    if widened:
        wq = i8.widen_weight_codes(wq)
    y = i8.linear(to_dev(x), wq, s_w, None if b is None else to_dev(b))
    i8.sync_check()
    return y


@pytest.mark.parametrize("M,N,K,bias", [
    (64, 128, 256, True),        # tiny config
    (1, 8, 16, True),
    (7, 24, 48, False),
    (129, 136, 272, True),
    (300, 200, 1040, False),
    (16, 3072, 12288, True),     # split-K path with the bf16 epilogue
    (2, 9216, 3072, True),
])
def test_linear_bf16_matches_oracle(orc, M, N, K, bias):
    shape = inputs.LinearShape("t", M, K, N, seed=M + N + K, outliers=K >= 256)
    d = inputs.linear_inputs(shape, with_bias=bias)
    y = _gpu_linear(d["x"], d["w"], d["bias"])
    want = _oracle_linear_rows(orc, d["x"], d["w"], d["bias"], np.arange(M))
    assert_bf16_exact(gpu_bf16_bits(y), want, f"{M}x{N}x{K}")


def test_widened_weights_bit_identical(orc):
    d = inputs.linear_inputs(inputs.LinearShape("w16", 300, 1040, 200, seed=9))
    y8 = _gpu_linear(d["x"], d["w"], d["bias"], widened=False)
    y16 = _gpu_linear(d["x"], d["w"], d["bias"], widened=True)
    assert torch.equal(y8.view(torch.int16), y16.view(torch.int16))


def test_zero_rows_give_bias(orc):
    M, N, K = 5, 64, 128
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[2] = 1.0
    w = inputs.random_bf16(N, K, seed=3, std=0.02)
    b = inputs.random_bf16(1, N, seed=4, std=0.5)[0]
    y = _gpu_linear(x, w, b)
    yb = gpu_bf16_bits(y)
    bb = inputs.bits(b)
    for r in (0, 1, 3, 4):
        assert np.array_equal(yb[r], bb)


def test_error_paths():
    a = torch.zeros(64, 128, dtype=torch.int8, device="cuda")
    w = torch.zeros(64, 128, dtype=torch.int8, device="cuda")
    raw = torch.zeros(64 * 128 + 16, dtype=torch.int8, device="cuda")
    with pytest.raises(i8.I8Error) as e:
        i8.gemm_int32(raw[1:1 + 64 * 128].view(64, 128), w)
    assert e.value.status == 2
    # a split-K shape with a too-small workspace (32 tokens, K = 12288: the
    # tiled kernel with K splits)
    a2 = torch.zeros(32, 12288, dtype=torch.int8, device="cuda")
    w2 = torch.zeros(3072, 12288, dtype=torch.int8, device="cuda")
    need = i8.workspace_bytes(32, 3072, 12288)
    assert need > 0
    with pytest.raises(i8.I8Error) as e:
        i8.gemm_int32(a2, w2, workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4
    i8.sync_check()


def test_timeout_is_reported_without_fault():
    """A pipeline wait that nothing completes ends by its time limit; the
    status word reports it and the context stays usable."""
    lib = i8.load()
    import ctypes
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.i8_selftest_timeout(50, s) == 0
    with pytest.raises(i8.I8Error) as e:
        i8.sync_check()
    assert e.value.status == 6
    i8.sync_check()  # cleared
    a = torch.ones(64, 64, dtype=torch.int8, device="cuda")
    c = i8.gemm_int32(a, a)
    i8.sync_check()
    assert int(c[0, 0]) == 64


@pytest.fixture
def cta_pair_option():
    yield
    i8.set_option("cta_pair", 0)


@pytest.mark.parametrize("mode", [1, 2], ids=["single_cta", "cta_pair"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 264, 1040), (520, 776, 4096)])
def test_gemm_int32_both_kernels(orc, cta_pair_option, mode, M, N, K):
    """Both GEMM kernels (one CTA per tile, and CTA pairs with 256 x 256
    tiles) on ragged shapes, random and adversarial operands."""
    i8.set_option("cta_pair", mode)
    a = inputs.random_int8(M, K, seed=M + 7 * K)
    w = inputs.random_int8(N, K, seed=N + 11 * K)
    a[:3], w[:3] = _adversarial(3, 3, K, seed=M)[0], _adversarial(3, 3, K, seed=N)[1]
    c = i8.gemm_int32(to_dev(a), to_dev(w))
    i8.sync_check()
    got = c.cpu().numpy()
    want = orc.gemm_s32(a.numpy(), w.numpy())
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"mode {mode}: {len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("M,N,K,splits", [(1, 200, 8192, 0), (16, 520, 8192, 0), (9, 64, 131072, 0),
                                           (1, 200, 8192, 1), (16, 520, 8192, 1), (3, 64, 6144, 1)])
def test_skinny_kernel_adversarial_exact(orc, M, N, K, splits):
    """Few tokens take the weight-streaming kernel (forced up to M = 16 here):
    each warp's fp32 accumulators gather 16-K MMA partials over 8 stages (16
    partials of at most 16 * 127^2 for +-127 operands, < 2^22) and drain into
    int32, then integer adds across warps and K splits.  One split: whole
    drain windows in one CTA (8192 K: four; 6144 K: two and a short one)."""
    a, w = _adversarial(max(M, 4), N, K, seed=M + N)
    a = a[:M].contiguous()
    i8.set_option("skinny_max_m", 16)
    i8.set_option("force_splits", splits)
    try:
        assert i8.plan_query(M, N, K, "int8")["kernel"] == "skinny"
        if splits:
            assert i8.plan_query(M, N, K, "int8")["splits"] == splits
        c = i8.gemm_int32(to_dev(a), to_dev(w))
        i8.sync_check()
    finally:
        i8.set_option("skinny_max_m", SKINNY_DEFAULT)
        i8.set_option("force_splits", 0)
    got = c.cpu().numpy()
    want = orc.gemm_s32(a.numpy(), w.numpy())
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("M", [1, 5, 16])
def test_skinny_kernel_widened_weights_and_off_switch(orc, M):
    shape = inputs.LinearShape("sk", M, 3072, 9216, seed=40 + M)
    d = inputs.linear_inputs(shape)
    rows = np.arange(M)
    want = _oracle_linear_rows(orc, d["x"], d["w"], d["bias"], rows)
    i8.set_option("skinny_max_m", 16)  # the weight-streaming kernel, forced up to M = 16
    try:
        y16 = _gpu_linear(d["x"], d["w"], d["bias"], widened=True)
    finally:
        i8.set_option("skinny_max_m", SKINNY_DEFAULT)
    assert_bf16_exact(gpu_bf16_bits(y16), want, "skinny w16")
    i8.set_option("skinny_max_m", 0)   # the tiled kernels for the same shape
    try:
        y8 = _gpu_linear(d["x"], d["w"], d["bias"], widened=False)
    finally:
        i8.set_option("skinny_max_m", SKINNY_DEFAULT)
    assert_bf16_exact(gpu_bf16_bits(y8), want, "tiled")


@pytest.mark.parametrize("M,N,K", [(512, 512, 1024), (130, 144, 272), (2, 9216, 3072), (5, 256, 512)],
                         ids=["cta_pair", "single_cta", "skinny_split", "skinny"])
def test_dependent_launches_keep_stream_order(M, N, K):
    """Kernels are scheduled while the previous kernel drains; each one waits
    for the previous kernel's memory before touching global memory.  A chain
    that reuses every buffer at once (codes, scales, workspace overwritten by
    the next call; a GEMM output quantized as the next layer's input) run
    back to back without host syncs must give the results of the same chain
    run one call at a time with plain launches."""
    g = torch.Generator().manual_seed(M + N + K)
    xs = [inputs.activations(M, K, g, "normal", True).cuda() for _ in range(3)]
    w1 = inputs.random_bf16(N, K, seed=5, std=0.02).cuda()
    w2 = inputs.random_bf16(K, N, seed=6, std=0.02).cuda()
    b1 = inputs.random_bf16(1, N, seed=7, std=0.1)[0].cuda()
    w1q, s1 = i8.quant_weight_perchannel(w1)
    w2q, s2 = i8.quant_weight_perchannel(w2)
    codes = torch.empty(M * max(K, N), dtype=torch.int8, device="cuda")   # shared by both layers
    sa = torch.empty(M, dtype=torch.float32, device="cuda")
    ws_bytes = max(i8.workspace_bytes(M, N, K), i8.workspace_bytes(M, K, N), 16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

    def chain(sync):
        outs = []
        for x in xs:
            a = codes[:M * K].view(M, K)
            i8.quant_act_pertoken(x, a, sa)
            if sync:
                torch.cuda.synchronize()
            y = i8.gemm_dequant_bias_bf16(a, sa, w1q, s1, b1, workspace=ws)
            if sync:
                torch.cuda.synchronize()
            a2 = codes[:M * N].view(M, N)
            i8.quant_act_pertoken(y, a2, sa)       # the GEMM output is the next input
            if sync:
                torch.cuda.synchronize()
            z = i8.gemm_dequant_bias_bf16(a2, sa, w2q, s2, None, workspace=ws)
            if sync:
                torch.cuda.synchronize()
            outs += [y, z]
        torch.cuda.synchronize()
        return [o.clone() for o in outs]

    try:
        i8.set_option("pdl", 0)
        want = chain(sync=True)
        i8.set_option("pdl", 1)
        for _ in range(5):
            got = chain(sync=False)
            for a, b in zip(got, want):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    finally:
        i8.set_option("pdl", 1)


@pytest.fixture
def stream_k_option():
    yield
    i8.set_option("stream_k", 1)
    i8.set_option("cta_pair", 0)


# Shapes on CTA pairs whose whole tiles leave pairs idle, so the stream-K
# schedule splits tiles between pairs: 2 x 3 tiles spread over many pairs
# (each tile shared by several), a ragged one, a multi-wave one with a
# partial last wave, and two with K >= 64 blocks, whose schedule runs one
# whole wave of 76 (or 74) tiles first and splits only the 5 (or 7) left
# over (ragged M, N and K in the second).
STREAM_K_SHAPES = [(512, 768, 4096), (300, 520, 1040), (1280, 2816, 2048), (2304, 2304, 8192),
                   (2200, 2104, 8208)]


@pytest.mark.parametrize("M,N,K", STREAM_K_SHAPES)
def test_stream_k_int32_exact(orc, stream_k_option, M, N, K):
    """Tiles finished from int32 partials of several pairs are bit-exact,
    adversarial rows included (partials near the int32 range)."""
    i8.set_option("cta_pair", 2)
    i8.set_option("stream_k", 2)
    a = inputs.random_int8(M, K, seed=M + 3 * K)
    w = inputs.random_int8(N, K, seed=N + 5 * K)
    a[:3], w[:3] = _adversarial(3, 3, K, seed=M)[0], _adversarial(3, 3, K, seed=N)[1]
    c = i8.gemm_int32(to_dev(a), to_dev(w))
    i8.sync_check()
    got = c.cpu().numpy()
    want = orc.gemm_s32(a.numpy(), w.numpy())
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("M,N,K", STREAM_K_SHAPES)
def test_stream_k_matches_whole_tiles(stream_k_option, M, N, K):
    """The bf16 output with the stream-K schedule equals the whole-tile
    schedule's bit for bit (both exact in int32, same epilogue)."""
    i8.set_option("cta_pair", 2)
    g = torch.Generator().manual_seed(M + N)
    x = inputs.activations(M, K, g, "normal", True).cuda()
    w = inputs.random_bf16(N, K, seed=N + K, std=0.02).cuda()
    b = inputs.random_bf16(1, N, seed=K, std=0.1)[0].cuda()
    wq, s_w = i8.quant_weight_perchannel(w)
    i8.set_option("stream_k", 0)
    want = i8.linear(x, wq, s_w, b)
    i8.set_option("stream_k", 2)
    got = i8.linear(x, wq, s_w, b)
    i8.sync_check()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_stream_k_workspace_garbage_and_graph_replay(stream_k_option):
    """Arrival words are tagged per launch: a workspace full of random bytes,
    or of another shape's leftovers, and CUDA-graph replays of one captured
    launch (which reuse its tag) all give the exact result."""
    i8.set_option("cta_pair", 2)
    i8.set_option("stream_k", 2)
    M, N, K = 512, 768, 4096
    a = inputs.random_int8(M, K, seed=1).cuda()
    w = inputs.random_int8(N, K, seed=2).cuda()
    want = torch._int_mm(a, w.t())
    nbytes = max(i8.workspace_bytes(M, N, K), i8.workspace_bytes(1280, 2816, 2048))
    assert i8.workspace_bytes(M, N, K) > 0
    ws = torch.randint(-128, 128, (nbytes,), dtype=torch.int8, device="cuda").view(torch.uint8)
    out = torch.empty(M, N, dtype=torch.int32, device="cuda")
    i8.gemm_int32(a, w, out=out, workspace=ws)
    i8.sync_check()
    assert torch.equal(out, want)
    # another shape through the same workspace, then this one again
    a2 = inputs.random_int8(1280, 2048, seed=3).cuda()
    w2 = inputs.random_int8(2816, 2048, seed=4).cuda()
    assert torch.equal(i8.gemm_int32(a2, w2, workspace=ws), torch._int_mm(a2, w2.t()))
    out.zero_()
    i8.gemm_int32(a, w, out=out, workspace=ws)
    i8.sync_check()
    assert torch.equal(out, want)
    # one launch captured in a graph and replayed
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            i8.gemm_int32(a, w, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    i8.sync_check()


@pytest.mark.parametrize("M,N,K,splits", [(2, 3072, 3072, 0), (5, 3072, 12288, 0), (1, 200, 8192, 8),
                                           (7, 520, 3584, 7), (3, 64, 1280, 3), (16, 136, 2560, 5)])
def test_skinny_cluster_splits_back_to_back_and_graph_replay(orc, M, N, K, splits):
    """The few-token kernel's K splits meet in the distributed shared memory
    of their cluster: no workspace, and back-to-back calls and CUDA-graph
    replays give the exact result.  Forced split counts up to the cluster
    limit of 8, odd ones (uneven shares of the outputs) and 16 tokens (two
    token groups) included."""
    a = inputs.random_int8(M, K, seed=M + 11)
    w = inputs.random_int8(N, K, seed=N + 12)
    want = orc.gemm_s32(a.numpy(), w.numpy())
    a, w = a.cuda(), w.cuda()
    i8.set_option("skinny_max_m", 16)
    i8.set_option("force_splits", splits)
    try:
        plan = i8.plan_query(M, N, K, "int8")
        assert plan["kernel"] == "skinny" and plan["ws_bytes"] == 0
        if splits:
            assert plan["splits"] == splits
        assert i8.workspace_bytes(M, N, K) == 0
        out = torch.empty(M, N, dtype=torch.int32, device="cuda")
        for _ in range(2):
            out.fill_(7)
            i8.gemm_int32(a, w, out=out)
            i8.sync_check()
            assert np.array_equal(out.cpu().numpy(), want)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                i8.gemm_int32(a, w, out=out)
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(3):
            out.fill_(7)
            graph.replay()
            torch.cuda.synchronize()
            assert np.array_equal(out.cpu().numpy(), want)
        i8.sync_check()
    finally:
        i8.set_option("skinny_max_m", SKINNY_DEFAULT)
        i8.set_option("force_splits", 0)


@pytest.fixture
def stage_k_option():
    yield
    i8.set_option("pair_stage_k", 0)
    i8.set_option("stream_k", 1)
    i8.set_option("cta_pair", 0)
    i8.set_option("chunk_k", 1024)


@pytest.mark.parametrize("stream_k", [0, 2])
@pytest.mark.parametrize("chunk_k", [1024, 384, 128])
@pytest.mark.parametrize("M,N,K", [(512, 768, 4096), (300, 520, 1040), (2560, 9216, 3072)])
def test_pair_stage_k_128_matches_64(orc, stage_k_option, stream_k, chunk_k, M, N, K):
    """The pair kernel with one fp16 stage per 128 K (two 64-K sub-tiles)
    gives the 64-K-stage kernel's int32 sums bit for bit, with whole tiles and
    with stream-K, and with accumulator restarts every 128, 384 or 1024 K; the
    int32 sums are also checked against the oracle on the small shapes."""
    i8.set_option("cta_pair", 2)
    i8.set_option("stream_k", stream_k)
    i8.set_option("chunk_k", chunk_k)
    a = inputs.random_int8(M, K, seed=M + K + chunk_k)
    w = inputs.random_int8(N, K, seed=N + K)
    a[:3], w[:3] = _adversarial(3, 3, K, seed=M)[0], _adversarial(3, 3, K, seed=N)[1]
    res = {}
    for sk in (64, 128):
        i8.set_option("pair_stage_k", sk)
        res[sk] = i8.gemm_int32(to_dev(a), to_dev(w))
        i8.sync_check()
    assert torch.equal(res[64], res[128])
    if M * N <= 512 * 768:
        assert np.array_equal(res[128].cpu().numpy(), orc.gemm_s32(a.numpy(), w.numpy()))


def test_pair_stage_k_option_values():
    assert i8.get_option("pair_stage_k") == 0
    for bad in (32, 96, 256, -1):
        with pytest.raises(i8.I8Error):
            i8.set_option("pair_stage_k", bad)
    i8.set_option("pair_stage_k", 64)
    assert i8.get_option("pair_stage_k") == 64
    i8.set_option("pair_stage_k", 0)


@pytest.fixture
def raster_option():
    yield
    i8.set_option("raster", 0)
    i8.set_option("stream_k", 1)
    i8.set_option("cta_pair", 0)


@pytest.mark.parametrize("route", ["int8", "int8_stream_k", "e4m3", "f16codes"])
@pytest.mark.parametrize("M,N,K", [(1280, 520, 2048), (300, 1040, 1040), (2560, 768, 4096)])
def test_tile_order_does_not_change_results(raster_option, route, M, N, K):
    """M-blocks-fastest and N-blocks-fastest tile orders give the same bits on
    every route (ragged edges, split-K and stream-K included)."""
    g = torch.Generator().manual_seed(M + N + K)
    x = inputs.activations(M, K, g, "normal", True).cuda()
    w = inputs.random_bf16(N, K, seed=N + K, std=0.02).cuda()
    b = inputs.random_bf16(1, N, seed=K, std=0.1)[0].cuda()
    if route == "int8_stream_k":
        i8.set_option("cta_pair", 2)
        i8.set_option("stream_k", 2)
    outs = []
    for order in (1, 2):
        i8.set_option("raster", order)
        if route.startswith("int8"):
            wq, s_w = i8.quant_weight_perchannel(w)
            y = i8.linear(x, wq, s_w, b)
        elif route == "e4m3":
            wq, s_w = i8.quant_weight_perchannel_e4m3(w)
            y = i8.linear_e4m3(x, wq, s_w, b)
        else:
            wq, s_w = i8.quant_weight_perchannel(w)
            y = i8.linear_f16codes(x, i8.widen_weight_codes(wq), s_w, b)
        i8.sync_check()
        outs.append(y.view(torch.int16))
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("route", ["int8", "f16codes", "e4m3", "layernorm", "gelu"])
def test_empty_token_batch(route):
    """No tokens: every route returns an empty [0, N] output (and empty codes
    and scales), with no launch failure and no device error."""
    K, N = 256, 128
    x = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    w = inputs.random_bf16(N, K, seed=1, std=0.02).cuda()
    b = inputs.random_bf16(1, N, seed=2, std=0.1)[0].cuda()
    if route == "int8":
        wq, s_w = i8.quant_weight_perchannel(w)
        y = i8.linear(x, wq, s_w, b)
        q, s = i8.quant_act_pertoken(x)
        assert q.shape == (0, K) and s.shape == (0,)
    elif route == "f16codes":
        wq, s_w = i8.quant_weight_perchannel(w)
        y = i8.linear_f16codes(x, i8.widen_weight_codes(wq), s_w, b)
    elif route == "e4m3":
        wq, s_w = i8.quant_weight_perchannel_e4m3(w)
        y = i8.linear_e4m3(x, wq, s_w, b)
    else:
        fn = i8.layernorm_quant_act_pertoken if route == "layernorm" else i8.gelu_quant_act_pertoken
        q, s = fn(x)
        y = q
        assert s.shape == (0,)
    i8.sync_check()
    assert y.shape[0] == 0


@pytest.mark.parametrize("route", ["int8", "e4m3", "f16codes"])
def test_output_beyond_two_to_the_31_elements(orc, route):
    """Y with 65536 x 32768 = 2^31 elements (4 GiB of bf16): offsets past the
    32-bit range.  Sampled rows, the last row and the last column included,
    match the oracle bit for bit (exact routes) or within the bound (E4M3)."""
    M, N, K = 65536, 32768, 16
    g = torch.Generator().manual_seed(7)
    x = inputs.activations(M, K, g, "normal", False)
    w = inputs.random_bf16(N, K, seed=8, std=0.02)
    b = inputs.random_bf16(1, N, seed=9, std=0.1)[0]
    xd, wd, bd = to_dev(x), to_dev(w), to_dev(b)
    if route == "e4m3":
        wq, s_w = i8.quant_weight_perchannel_e4m3(wd)
        y = i8.linear_e4m3(xd, wq, s_w, bd)
    else:
        wq, s_w = i8.quant_weight_perchannel(wd)
        y = (i8.linear(xd, wq, s_w, bd) if route == "int8"
             else i8.linear_f16codes(xd, i8.widen_weight_codes(wq), s_w, bd))
    i8.sync_check()
    rows = np.array([0, 1, 32767, 32768, 65534, 65535])
    got = y[torch.from_numpy(rows).cuda()].cpu().view(torch.int16).numpy().view(np.uint16)
    del y
    torch.cuda.empty_cache()
    if route == "e4m3":
        ref = orc.linear_e4m3(inputs.bits(x[rows]), inputs.bits(w), inputs.bits(b))["y"]
        r = (ref.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        gg = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.all(np.abs(gg - r) <= 2.0 ** -6 * np.abs(r) + 1e-5)
    else:
        ref = orc.linear(inputs.bits(x[rows]), inputs.bits(w), inputs.bits(b))["y"]
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(2, 9216, 3072), (16, 3072, 12288), (300, 200, 1040),
                                   (512, 3072, 12288), (2304, 3072, 12288), (8704, 9216, 3072)])
def test_plan_query_on_the_device_matches_the_workspace_queries(M, N, K):
    """i8_plan_query with the current device's figures reports the workspace
    that each route's *_workspace_bytes asks for."""
    p8 = i8.plan_query(M, N, K, "int8")
    p16 = i8.plan_query(M, N, K, "w16")
    assert i8.workspace_bytes(M, N, K) == max(p8["ws_bytes"], p16["ws_bytes"])
    assert i8.e4m3_workspace_bytes(M, N, K) == i8.plan_query(M, N, K, "e4m3")["ws_bytes"]
    assert i8.f16codes_workspace_bytes(M, N, K) == i8.plan_query(M, N, K, "f16codes")["ws_bytes"]
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    for p in (p8, p16):
        if p["kernel"] != "skinny":          # tiled grids: at most one CTA per SM
            assert p["grid"] <= sms
