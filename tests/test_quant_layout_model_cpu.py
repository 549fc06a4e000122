"""The per-row quantizer's work split, modelled on the CPU for every K.

The quantizer ("Realizing Native INT8 Compute for Diffusion Transformers on
Consumer GPUs", abstract: one scale per token row) keeps a whole row in
registers: G warps share a row, each lane holds up to V 16-byte vectors (8
bf16 each), and lane `lane` of warp `wig` in the row's group owns the
vectors starting at element  wig * 256 * V + (i * 32 + lane) * 8,  i < V,
skipping those at or past K.  The host picks G (doubling from 1 while a
lane would need more than quant_vpl vectors, up to 8), V (the smallest
compiled size >= the vectors needed) and R rows per CTA (G * R <= 8 warps);
rows over 32768 elements go to a two-pass kernel.  This model checks, for
every K the library accepts up to that limit and every quant_vpl and
quant_rows option, that each element of the row is loaded and quantized by
exactly one lane, that no load runs past the row, and that a CTA stays within
256 threads.  A last test ties the model to the sources.
"""
import os

import numpy as np
import pytest

V_SIZES = [1, 2, 3, 4, 6, 8, 12, 16]


def host_choice(K, vpl, rows_opt):
    vecs = K // 8
    G = 1
    while G < 8 and -(-vecs // (32 * G)) > vpl:
        G *= 2
    need = -(-vecs // (32 * G))
    if need > 16:
        return None                                   # the two-pass kernel
    V = next(v for v in V_SIZES if need <= v)
    R = min(rows_opt, 8 // G) if rows_opt > 0 else 1
    return G, V, R


_STARTS = {}


def _starts(G, V):
    """Sorted first elements of every lane's vectors for a (G, V) launch
    (independent of K; the kernel masks those at or past K)."""
    if (G, V) not in _STARTS:
        _STARTS[(G, V)] = np.sort(np.array(
            [wig * 256 * V + (i * 32 + lane) * 8
             for wig in range(G) for i in range(V) for lane in range(32)]))
    return _STARTS[(G, V)]


@pytest.mark.parametrize("vpl", list(range(1, 17)))
def test_every_element_is_owned_by_exactly_one_lane(vpl):
    for K in range(16, 32768 + 1, 16):
        for rows_opt in (0, 1, 3, 8):
            G, V, R = host_choice(K, vpl, rows_opt)
            assert G in (1, 2, 4, 8) and 1 <= R and G * R <= 8
            assert 32 * G * R <= 256
        st = _starts(G, V)
        assert len(np.unique(st)) == len(st)              # no two lanes share a vector
        owned = st[st < K]
        assert np.array_equal(owned, np.arange(0, K, 8)), (vpl, K)
        assert owned[-1] + 8 <= K                         # no load past the row


def test_long_rows_go_to_the_two_pass_kernel():
    for vpl in (1, 6, 16):
        assert host_choice(32768, vpl, 0) is not None
        assert host_choice(32768 + 16, vpl, 0) is None
        assert host_choice(131072, vpl, 0) is None


def test_model_restates_the_sources():
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "w8a8_int8_quantized_i8_gb300", "csrc")

    def code(name):
        with open(os.path.join(root, name)) as fh:
            return " ".join(fh.read().split())

    api, quant = code("i8_api.cu"), code("quant.cuh")
    for text in ["const int vecs = static_cast<int>(K / 8); int G = 1; "
                 "while (G < 8 && (vecs + 32 * G - 1) / (32 * G) > g_opt.quant_vpl) G *= 2; "
                 "const int need = (vecs + 32 * G - 1) / (32 * G);",
                 "const int R = g_opt.quant_rows > 0 ? std::min(g_opt.quant_rows, 8 / G) : 1;",
                 "if (need > 16) {"]:
        assert text in api, text
    for v in V_SIZES[:-1]:
        assert f"if (need <= {v}) e = launch_quant_v<{v}>(" in api
    assert "e = launch_quant_v<16>(" in api
    for text in ["const int slice0 = wig * (32 * 8 * V);",
                 "const int e = slice0 + (i * 32 + lane) * 8; if (valid_row && e < K) {"]:
        assert text in quant, text


def test_layernorm_producer_uses_the_same_split():
    """The LayerNorm producer-quantizer (one row per CTA of G warps) takes
    the same host choice of G and V and the same element index, and accepts
    only K <= 32768, so the coverage checked above holds for it too."""
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "w8a8_int8_quantized_i8_gb300", "csrc")

    def code(name):
        with open(os.path.join(root, name)) as fh:
            return " ".join(fh.read().split())

    api, prod = code("i8_api.cu"), code("producer.cuh")
    assert "if (K % 16 != 0 || K > 32768 || rows > INT32_MAX) return I8_ERR_UNSUPPORTED;" in api
    assert api.count("while (G < 8 && (vecs + 32 * G - 1) / (32 * G) > g_opt.quant_vpl) G *= 2;") == 2
    for v in V_SIZES[:-1]:
        assert f"if (need <= {v}) return launch_producer_v<{v}, FMT>(" in api
    assert "return launch_producer_v<16, FMT>(" in api
    assert "const int slice0 = warp * (32 * 8 * V);" in prod
    assert "const int e = slice0 + (i * 32 + lane) * 8;" in prod
    for vpl in range(1, 17):
        for K in (16, 3072, 12288, 32768):
            G, V, _ = host_choice(K, vpl, 0)
            owned = _starts(G, V)[_starts(G, V) < K]
            assert np.array_equal(owned, np.arange(0, K, 8))


def test_gelu_kernel_row_walk_with_prefetch():
    """The GELU producer walks groups of R rows with a grid stride and, for
    rows of at most 8 vectors per lane, loads the next group before
    processing the current one.  Simulated for many row counts, grids and R:
    every row is processed exactly once, from the data loaded for that row."""
    for rows in (1, 2, 7, 8, 9, 100, 1023, 4096):
        for grid in (1, 3, 152, 304):
            for R in (1, 2, 4, 8):
                for prefetch in (True, False):
                    stride = grid * R
                    done = []
                    for blk in range(grid):
                        base = blk * R
                        cur = base if (prefetch and base < rows) else None
                        while base < rows:
                            nxt = base + stride if (prefetch and base + stride < rows) else None
                            if not prefetch:
                                cur = base
                            assert cur == base             # the loaded group is this group
                            done.extend(r for r in range(base, base + R) if r < rows)
                            cur = nxt
                            base += stride
                    assert sorted(done) == list(range(rows))
    src_path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "w8a8_int8_quantized_i8_gb300", "csrc", "producer.cuh")
    with open(src_path) as fh:
        src = " ".join(fh.read().split())
    for text in ["const int64_t stride = static_cast<int64_t>(gridDim.x) * R;",
                 "int64_t base = static_cast<int64_t>(blockIdx.x) * R;",
                 "if (kPrefetch && base < rows) load_rows(base, v);",
                 "for (; base < rows; base += stride) {",
                 "if (base + stride < rows) load_rows(base + stride, vn);",
                 "for (int i = 0; i < V; ++i) v[i] = vn[i];"]:
        assert text in src, text
