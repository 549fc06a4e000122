"""Source guards for the properties the bit-exact epilogue depends on.

The epilogue computes bf16(((float(acc) * s_a) * s_w) + bias) with each step
an fp32 operation rounded to nearest even ("Realizing Native INT8 Compute for
Diffusion Transformers on Consumer GPUs", abstract: per-token x per-channel
dequantization and bias folded into the epilogue, bf16 out; the oracle's
reading fixes the order).  The GPU matches the oracle bit for bit only while
  * every epilogue goes through dequant_one, whose steps are the scalar
    __int2float_rn / __fmul_rn / __fadd_rn intrinsics (never contracted into
    an FMA; packed f32x2 multiply + add once were, one bf16 ulp off where the
    product and the bias nearly cancel), then a round-to-nearest bf16 cast;
  * no GEMM source uses packed f32x2 or fma arithmetic;
  * the build keeps IEEE fp32 behaviour (no flush to zero, correctly rounded
    division, no fast-math).
These checks read the sources only; the GPU parity tests check the results.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "w8a8_int8_quantized_i8_gb300", "csrc")
GEMM_SOURCES = ["gemm.cuh", "gemm_pair.cuh", "gemm_direct.cuh", "skinny.cuh"]


def _code(name):
    """The source with comments removed and whitespace collapsed."""
    with open(os.path.join(CSRC, name)) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def test_dequant_steps_are_the_scalar_rounded_intrinsics():
    src = _code("gemm.cuh")
    assert ("float dequant_one(int acc, float sa, float sw, float b) { "
            "float t = __int2float_rn(acc); t = __fmul_rn(t, sa); t = __fmul_rn(t, sw); "
            "return __fadd_rn(t, b); }") in src
    assert ("float dequant_one(float acc, float sa, float sw, float b) { "
            "float t = __fmul_rn(acc, sa); t = __fmul_rn(t, sw); return __fadd_rn(t, b); }") in src


def test_every_bf16_epilogue_goes_through_dequant_one():
    total = 0
    for name in GEMM_SOURCES:
        src = _code(name)
        # bf16 conversions in the GEMM sources take dequant_one's result,
        # either directly or through pack_bf16x2 of two dequant_one results
        for m in re.finditer(r"__float2bfloat16_rn\(([^;]*)\);", src):
            assert m.group(1).startswith("dequant_one("), (name, m.group(0))
            total += 1
        for m in re.finditer(r"pack_bf16x2\((\w+), (\w+)\);", src):
            for var in m.groups():
                assert re.search(rf"\b{var} = dequant_one\(", src), (name, var)
            total += 1
    assert total >= 5


def test_no_packed_or_fused_arithmetic_in_the_gemm_sources():
    for name in GEMM_SOURCES:
        src = _code(name)
        for pat in (r"f32x2", r"\bfma\.", r"__fmaf?_r", r"\bfmaf?\(", r"__fmul2", r"__fadd2"):
            assert not re.search(pat, src), (name, pat)


def test_build_keeps_ieee_fp32():
    from w8a8_int8_quantized_i8_gb300 import build
    flags = build.NVCC_FLAGS
    for f in ("-ftz=false", "-prec-div=true", "-prec-sqrt=true"):
        assert f in flags
    assert not any(f in ("--use_fast_math", "-use_fast_math") or f.startswith("-ftz=true")
                   for f in flags)
    assert "arch=compute_103a,code=sm_103a" in flags


KERNEL_SOURCES = ["gemm.cuh", "gemm_pair.cuh", "gemm_direct.cuh", "skinny.cuh", "quant.cuh",
                  "producer.cuh", "ptx.cuh", "i8_api.cu"]


def test_every_pipeline_wait_is_bounded():
    """Raw mbarrier polls appear only inside the bounded wait helpers, each of
    which gives up after a time limit (2 s) with the abort flag and the
    device status word set; no kernel source has another unbounded loop."""
    ptx = _code("ptx.cuh")
    assert "constexpr unsigned long long kWaitLimitNs = 2000000000ull;" in ptx
    helpers = {}
    for name in ("mbar_wait", "mbar_wait_bounded", "mbar_wait_cluster"):
        m = re.search(rf"bool {name}\((.*?)\) {{(.*?)\}} (?=__device__|//|$)", ptx)
        assert m, name
        helpers[name] = m.group(2)
        assert "globaltimer_ns() - t0 >" in m.group(2), name
        assert "return false;" in m.group(2) and "atomicOr(&g_status, 1u << 6);" in m.group(2)
    for name in KERNEL_SOURCES:
        src = _code(name)
        # every raw poll sits inside a helper body
        polls = len(re.findall(r"\bmbar_try_wait(?:_cluster)?\(bar, parity\)", src))
        if name == "ptx.cuh":
            inside = sum(len(re.findall(r"\bmbar_try_wait(?:_cluster)?\(bar, parity\)", b))
                         for b in helpers.values())
            assert polls == inside
        else:
            assert "mbar_try_wait" not in src, name
        # no other unbounded loop shapes in device code
        if name != "i8_api.cu":
            assert "for (;;)" not in src and "do {" not in src, name
            if name != "ptx.cuh":
                assert not re.search(r"\bwhile\s*\(", src), name


def test_stream_k_arrival_loop_is_capped():
    src = _code("gemm_pair.cuh")
    m = re.search(r"bool sk_arrive\((.*?)\) \{(.*?)\n?\}", src)
    assert m and "for (int i = 0; i < 4096; ++i)" in m.group(2)


def test_no_device_code_traps_or_asserts():
    for name in KERNEL_SOURCES:
        src = _code(name)
        assert "__trap" not in src and "trap;" not in src, name
        assert not re.search(r"(?<!static_)\bassert\(", src), name


def test_tma_inner_coordinates_are_16_byte_multiples():
    """A tiled TMA copy must start its innermost coordinate on a 16-byte
    boundary.  Every x argument in the kernels is one of the expressions
    below, each a whole number of 128-byte rows: K-block starts (128 int8 /
    E4M3 codes, 64 fp16 codes, 256-code stages of 128- or 64-element boxes)
    and output column starts (64 bf16 or 32 int32 columns from a multiple of
    128), and the stream-K partial reloads (32 int32 columns from a multiple
    of 128)."""
    allowed_x = {"kb * Cfg::BK8", "k16", "kb * Cfg::BK", "k0 + b * Cfg::BOX_K", "k0 + b * Cfg::A_BOX_K",
                 "(ks0 + i) * kSkinnyK + b * Cfg::BOX_K", "(ks0 + i + Cfg::STAGES) * kSkinnyK + b * Cfg::BOX_K",
                 "nb", "n0 + g * 32", "n0 + g * 64", "n_loc + 32 * g"}
    calls = 0
    for name in GEMM_SOURCES:
        src = _code(name)
        for m in re.finditer(r"\b(tma_load_[23]d(?:_pair)?|tma_store_3d|tma_prefetch_l2_2d)\(([^;]*)\);",
                             src):
            args = [a.strip() for a in m.group(2).split(",")]
            x = (args[3] if m.group(1).startswith("tma_load")
                 else args[1] if m.group(1).startswith("tma_prefetch") else args[2])
            assert x in allowed_x, (name, m.group(0))
            calls += 1
    assert calls >= 12
    gemm, pair, skinny = _code("gemm.cuh"), _code("gemm_pair.cuh"), _code("skinny.cuh")
    direct = _code("gemm_direct.cuh")
    # the expressions' parts
    assert "static constexpr int BK8 = 128;" in gemm and "static constexpr int BK16 = 64;" in gemm
    assert "static constexpr int BK8 = 128;" in pair and "static constexpr int BK16 = 64;" in pair
    assert "static constexpr int BK = KIND == kDirectF16 ? 64 : 128;" in direct
    assert "constexpr int kSkinnyK = 256;" in skinny
    assert "const int k0 = (ks0 + i) * kSkinnyK;" in skinny
    assert "static constexpr int BOX_K = W_F16 ? 64 : 128;" in skinny
    assert "static constexpr int A_BOX_K = A_F16 ? 64 : 128;" in skinny
    assert "const int k16 = kb * Cfg::BK8 + h * Cfg::BK16;" in gemm
    assert "const int k16 = kb * Cfg::BK8 + (h + q) * Cfg::BK16;" in pair
    assert "const int nb = n0 + g * 64;" in gemm
    # output column starts passed to the store helpers: multiples of 128
    for src, expr in ((gemm, "tc.nb * Cfg::BN + cg * 128"),
                      (direct, "const int n_base = t.nb * Cfg::PAIR_N + cg * 128;"),
                      (pair, "const int n_loc = cg * 128;")):
        assert expr in src, expr
    # the staged-scale store starts its 64-column groups at the callers' n0:
    # a tile column base plus n_loc, a multiple of 128 bf16 columns
    assert "tc.nb * Cfg::PAIR_N + n_loc, acc, sa," in pair
    assert "n_sub" not in pair
