"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every function include/i8.h declares, and rejects bad
arguments on the host before touching a device."""
import ctypes

import pytest

from w8a8_int8_quantized_i8_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_every_declared_function_is_exported(lib):
    names = binding.header_functions()
    assert len(names) >= 12
    for n in ["i8_quant_weight_perchannel", "i8_quant_act_pertoken", "i8_gemm_int32",
              "i8_gemm_dequant_bias_bf16", "i8_gemm_workspace_bytes", "i8_sync_check"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for code, name in binding.STATUS.items():
        assert lib.i8_status_string(code).decode() == name
    assert lib.i8_status_string(99).decode() == "I8_ERR_UNKNOWN"
    assert b"sm_103a" in lib.i8_version()


P = ctypes.c_void_p


def test_quant_argument_errors(lib):
    ok = P(0x10000)
    for fn in (lib.i8_quant_act_pertoken, lib.i8_quant_weight_perchannel):
        assert fn(ok, -1, 64, 64, ok, 64, ok, None) == 1            # negative rows
        assert fn(ok, 4, 64, 32, ok, 64, ok, None) == 1             # ldx < K
        assert fn(None, 4, 64, 64, ok, 64, ok, None) == 1           # NULL input
        assert fn(ok, 4, 40, 40, ok, 48, ok, None) == 3             # K % 16
        assert fn(ok, 4, 131072 + 16, 131072 + 16, ok, 131088, ok, None) == 3
        assert fn(P(0x10008), 4, 64, 64, ok, 64, ok, None) == 2     # misaligned x
        assert fn(ok, 4, 64, 68, ok, 64, ok, None) == 2             # row stride
        assert fn(ok, 0, 64, 64, ok, 64, ok, None) == 0             # empty: no-op


def test_gemm_argument_errors(lib):
    ok = P(0x10000)
    g = lib.i8_gemm_dequant_bias_bf16
    assert g(ok, ok, ok, ok, None, -1, 8, 16, ok, 8, None, 0, None) == 1
    assert g(ok, ok, ok, ok, None, 4, 8, 24, ok, 8, None, 0, None) == 3     # K % 16
    assert g(ok, ok, ok, ok, None, 0, 8, 16, ok, 8, None, 0, None) == 0     # empty
    assert g(None, ok, ok, ok, None, 4, 8, 16, ok, 8, None, 0, None) == 1
    assert g(ok, None, ok, ok, None, 4, 8, 16, ok, 8, None, 0, None) == 1   # no scales
    assert g(P(0x10001), ok, ok, ok, None, 4, 8, 16, ok, 8, None, 0, None) == 2
    assert g(ok, ok, ok, P(0x10004), None, 4, 8, 16, ok, 8, None, 0, None) == 2  # s_w
    assert g(ok, ok, ok, ok, P(0x10002), 4, 8, 16, ok, 8, None, 0, None) == 2    # bias
    assert g(ok, ok, ok, ok, None, 4, 12, 16, ok, 12, None, 0, None) == 2        # ldy % 8
    c = lib.i8_gemm_int32
    assert c(ok, ok, 4, 8, 16, ok, 6, None, 0, None) == 1                   # ldc < N
    assert c(ok, ok, 4, 8, 16, ok, 10, None, 0, None) == 2                  # ldc % 4
    assert c(ok, ok, 4, 8, 200000, ok, 8, None, 0, None) == 3
    assert lib.i8_widen_weight_codes(ok, 4, 24, ok, None) == 3


def test_e4m3_argument_errors(lib):
    ok = P(0x10000)
    for fn in (lib.i8_quant_act_pertoken_e4m3, lib.i8_quant_weight_perchannel_e4m3):
        assert fn(ok, -1, 64, 64, ok, 64, ok, None) == 1
        assert fn(ok, 4, 40, 40, ok, 48, ok, None) == 3             # K % 16
        assert fn(P(0x10008), 4, 64, 64, ok, 64, ok, None) == 2
        assert fn(ok, 0, 64, 64, ok, 64, ok, None) == 0
    g = lib.i8_gemm_e4m3_dequant_bias_bf16
    assert g(ok, ok, ok, ok, None, -1, 8, 16, ok, 8, None, 0, None) == 1
    assert g(ok, ok, ok, ok, None, 4, 8, 24, ok, 8, None, 0, None) == 3    # K % 16
    assert g(ok, ok, ok, ok, None, 0, 8, 16, ok, 8, None, 0, None) == 0    # empty
    assert g(ok, None, ok, ok, None, 4, 8, 16, ok, 8, None, 0, None) == 1  # no scales
    assert g(P(0x10001), ok, ok, ok, None, 4, 8, 16, ok, 8, None, 0, None) == 2
    assert g(ok, ok, ok, ok, None, 4, 12, 16, ok, 12, None, 0, None) == 2  # ldy % 8
    c = lib.i8_gemm_e4m3_f32
    assert c(ok, ok, 4, 8, 16, ok, 6, None, 0, None) == 1                  # ldc < N
    assert c(ok, ok, 4, 8, 16, ok, 10, None, 0, None) == 2                 # ldc % 4
    assert c(ok, ok, 4, 8, 200000, ok, 8, None, 0, None) == 3
    assert lib.i8_gemm_e4m3_workspace_bytes(4, 8, 24) == 0


def test_options_validation(lib):
    assert lib.i8_set_option(1, 100) == 1
    assert lib.i8_set_option(1, 2048) == 1
    assert lib.i8_set_option(1, 512) == 0
    assert lib.i8_set_option(2, -1) == 1
    assert lib.i8_set_option(2, 0) == 0
    assert lib.i8_set_option(77, 0) == 1
    assert lib.i8_set_option(8, 2) == 1           # PDL: 0 or 1
    assert lib.i8_set_option(8, 0) == 0
    assert lib.i8_set_option(8, 1) == 0
    assert lib.i8_set_option(9, 9) == 1           # quantizer rows per CTA: 0..8
    assert lib.i8_set_option(9, -1) == 1
    assert lib.i8_set_option(9, 0) == 0
    assert lib.i8_set_option(10, 3) == 1          # stream-K: 0, 1 or 2
    assert lib.i8_set_option(10, 2) == 0
    assert lib.i8_set_option(10, 0) == 0
    assert lib.i8_set_option(10, 1) == 0
    assert lib.i8_set_option(1, 1024) == 0        # restore the default chunk
    assert lib.i8_selftest_timeout(0, None) == 1


def test_get_option_and_nvtx_ranges(lib):
    v = ctypes.c_int64(-1)
    assert lib.i8_get_option(1, ctypes.byref(v)) == 0 and v.value == 1024
    assert lib.i8_get_option(77, ctypes.byref(v)) == 1
    assert lib.i8_get_option(1, None) == 1
    assert lib.i8_set_option(11, 1) == 0                  # NVTX ranges on
    assert lib.i8_get_option(11, ctypes.byref(v)) == 0 and v.value == 1
    # calls rejected on the host still open and close their range cleanly
    assert lib.i8_gemm_int32(P(0x10000), P(0x10000), 4, 8, 24, P(0x10000), 8, None, 0, None) == 3
    assert lib.i8_set_option(11, 2) == 1
    assert lib.i8_set_option(11, 0) == 0
    # K per fp16 stage of the pair kernel: 0 (by the chunk length), 64 or 128
    assert lib.i8_get_option(12, ctypes.byref(v)) == 0 and v.value == 0
    for bad in (1, 32, 96, 192, 256):
        assert lib.i8_set_option(12, bad) == 1
    assert lib.i8_set_option(12, 64) == 0
    assert lib.i8_get_option(12, ctypes.byref(v)) == 0 and v.value == 64
    assert lib.i8_set_option(12, 0) == 0
    # tile order: 0 (by shape), 1 M blocks fastest, 2 N blocks fastest
    assert lib.i8_get_option(13, ctypes.byref(v)) == 0 and v.value == 0
    assert lib.i8_set_option(13, 3) == 1 and lib.i8_set_option(13, -1) == 1
    assert lib.i8_set_option(13, 2) == 0 and lib.i8_set_option(13, 0) == 0


def test_options_from_the_environment(tmp_path):
    """I8_OPTIONS is read when the library loads; bad entries are ignored."""
    import subprocess
    import sys
    code = ("import ctypes, sys; sys.path.insert(0, %r); "
            "from w8a8_int8_quantized_i8_gb300 import binding; "
            "print(binding.get_option('chunk_k'), binding.get_option('stream_k'), "
            "binding.get_option('nvtx'), binding.get_option('pdl'))") % str(build.ROOT)
    env = dict(__import__("os").environ,
               I8_OPTIONS="chunk_k=512,stream_k=0,nvtx=1,pdl=7,bogus=3,tile_n=abc")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True).stdout.split()
    assert out == ["512", "0", "1", "1"]


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(OSError):
        binding.load(str(tmp_path / "missing_libi8.so"))


def test_workspace_query_rejects_bad_shapes(lib):
    assert lib.i8_gemm_workspace_bytes(4, 8, 24) == 0
    assert lib.i8_gemm_workspace_bytes(-4, 8, 16) == 0


def test_empty_inputs_are_no_ops(lib):
    """M = 0 (and N = 0 for the GEMMs) is a valid call that does nothing: each
    entry point returns I8_OK before touching a pointer or the device (this
    runs without a GPU, with null pointers)."""
    N0 = None
    K = 64
    calls = {
        "i8_quant_act_pertoken": lambda: lib.i8_quant_act_pertoken(N0, 0, K, K, N0, K, N0, N0),
        "i8_quant_weight_perchannel": lambda: lib.i8_quant_weight_perchannel(N0, 0, K, K, N0, K, N0, N0),
        "i8_quant_act_pertoken_e4m3": lambda: lib.i8_quant_act_pertoken_e4m3(N0, 0, K, K, N0, K, N0, N0),
        "i8_quant_weight_perchannel_e4m3": lambda: lib.i8_quant_weight_perchannel_e4m3(N0, 0, K, K, N0, K, N0, N0),
        "i8_quant_act_pertoken_f16codes": lambda: lib.i8_quant_act_pertoken_f16codes(N0, 0, K, K, N0, K, N0, N0),
        "i8_layernorm_quant_act_pertoken": lambda: lib.i8_layernorm_quant_act_pertoken(
            N0, 0, K, K, ctypes.c_float(1e-6), 0, N0, K, N0, N0, K, N0),
        "i8_gelu_quant_act_pertoken": lambda: lib.i8_gelu_quant_act_pertoken(N0, 0, K, K, 0, N0, K, N0, N0, K, N0),
        "i8_widen_weight_codes": lambda: lib.i8_widen_weight_codes(N0, 0, K, N0, N0),
    }
    for M, N in ((0, 8), (4, 0), (0, 0)):
        calls[f"i8_gemm_int32 {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_int32(N0, N0, M, N, K, N0, max(N, 1), N0, 0, N0)
        calls[f"i8_gemm_dequant_bias_bf16 {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_dequant_bias_bf16(
            N0, N0, N0, N0, N0, M, N, K, N0, max(N, 8), N0, 0, N0)
        calls[f"i8_gemm_dequant_bias_bf16_w16 {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_dequant_bias_bf16_w16(
            N0, N0, N0, N0, N0, M, N, K, N0, max(N, 8), N0, 0, N0)
        calls[f"i8_gemm_e4m3_f32 {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_e4m3_f32(N0, N0, M, N, K, N0, max(N, 4), N0, 0, N0)
        calls[f"i8_gemm_e4m3_dequant_bias_bf16 {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_e4m3_dequant_bias_bf16(
            N0, N0, N0, N0, N0, M, N, K, N0, max(N, 8), N0, 0, N0)
        calls[f"i8_gemm_int32_f16codes {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_int32_f16codes(
            N0, N0, M, N, K, N0, max(N, 4), N0, 0, N0)
        calls[f"i8_gemm_dequant_bias_bf16_f16codes {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_dequant_bias_bf16_f16codes(
            N0, N0, N0, N0, N0, M, N, K, N0, max(N, 8), N0, 0, N0)
        calls[f"i8_gemm_dequant_bias_bf16_noalloc {M}x{N}"] = lambda M=M, N=N: lib.i8_gemm_dequant_bias_bf16_noalloc(
            N0, N0, N0, N0, N0, M, N, K, N0, max(N, 8), N0)
    bad = {name: rc for name, rc in ((name, fn()) for name, fn in calls.items()) if rc != 0}
    assert not bad, bad


def test_option_tables_agree(lib, tmp_path):
    """The binding's option names and numbers are the header's i8_option enum,
    and every name is accepted through I8_OPTIONS when the library loads."""
    import os
    import re
    import subprocess
    import sys
    hdr = open(os.path.join(build.ROOT, "include", "i8.h")).read()
    enum = {m.group(1).lower(): int(m.group(2))
            for m in re.finditer(r"I8_OPT_([A-Z0-9_]+)\s*=\s*(\d+)", hdr)}
    assert enum == binding.OPTIONS
    # a value each option accepts that differs from its default
    probe = {"chunk_k": 512, "force_splits": 3, "max_ctas": 64, "tile_n": 128, "quant_vpl": 4,
             "cta_pair": 1, "skinny_max_m": 4, "pdl": 0, "quant_rows": 2, "stream_k": 0,
             "nvtx": 1, "pair_stage_k": 64, "raster": 2}
    assert set(probe) == set(binding.OPTIONS)
    env = dict(os.environ, I8_OPTIONS=",".join(f"{k}={v}" for k, v in probe.items()))
    code = ("import sys, json; sys.path.insert(0, %r); "
            "from w8a8_int8_quantized_i8_gb300 import binding; "
            "print(json.dumps({n: binding.get_option(n) for n in binding.OPTIONS}))") % str(build.ROOT)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True).stdout.strip().splitlines()[-1]
    import json
    assert json.loads(out) == probe


def test_every_compute_entry_point_cites_its_passage():
    """Each compute call in include/i8.h is documented by the comment block
    above it (or by its section's comment), and that text cites the passage
    that defines the operation, or says that the pages have none."""
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "i8.h")
    with open(hdr) as fh:
        text = fh.read()
    cites = re.compile(r"arXiv 2606\.14598|aiexpert\.news|OCP 8-bit|no counterpart|not on the pages|"
                       r"The pages (?:print|do not|never)", re.I)
    names = re.findall(r"^(?:i8_status|size_t)\s+(i8_[a-z0-9_]+)\(", text, re.M)
    compute = [n for n in names if re.search(r"quant|gemm|widen|layernorm|gelu", n)
               and not n.endswith("_workspace_bytes")]
    assert len(compute) >= 15
    missing = []
    for name in compute:
        pos = re.search(rf"^(?:i8_status|size_t)\s+{name}\(", text, re.M).start()
        # the nearest comment blocks above the declaration (its own and its section's)
        before = text[:pos]
        blocks = re.findall(r"/\*.*?\*/", before, re.S)
        assert blocks, name
        own = blocks[-1]
        section = next((b for b in reversed(blocks) if "----" in b), "")
        if not (cites.search(own) or cites.search(section)):
            missing.append(name)
    assert not missing, missing
