"""CPU checks of the C ABI: the library builds and loads, exports every symbol include/moe.h declares,
its host-side helpers are consistent, and bad arguments are rejected before any device work."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    import moe_expert_ffn_sqrt_gb300 as M
    if not os.path.exists(M.LIB_PATH):
        from moe_expert_ffn_sqrt_gb300 import build
        build.build()
    M.lib()
    return M


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(M):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(M.lib(), n), n


def test_sizes(M):
    assert M.msum_upper(8, 6, 256, 16) == 3888
    assert M.msum_upper(3, 2, 3, 1) == 6
    assert M.act_sf_block_rows(1) == 16 and M.act_sf_block_rows(64) == 64 and M.act_sf_block_rows(256) == 128
    # 256-row tiles: W13 [2, 512, 512] pairs rows (gate, up); W2 [2, 384, 256] has a half-empty last tile
    assert M.weight_packed_bytes("mxfp4", 2, 512, 512, 2) == 2 * 512 * (256 + 16)
    assert M.weight_packed_bytes("mxfp4", 2, 384, 256, 1) == 2 * 2 * 2 * 2 * (8192 + 512)
    assert M.weight_packed_bytes("mxfp4", 2, 384, 256, 2) == 0
    n = M.workspace_size(8, 7168, 2048, 256, 6, 16)
    assert n > 3888 * 7168  # holds the permuted activations


@pytest.mark.parametrize("rows,slabs,align", [(3888, 56, 16), (100, 2, 1), (257, 16, 64), (1000, 5, 256), (0, 4, 16)])
def test_act_sf_tile_roundtrip(M, rows, slabs, align):
    rng = np.random.default_rng(rows + slabs)
    plain = rng.integers(0, 256, size=(rows, slabs), dtype=np.uint8)
    tiled = M.act_sf_tile(plain, align)
    assert tiled.size == M.act_sf_tiled_bytes(rows, slabs, align)
    assert np.array_equal(M.act_sf_untile(tiled, rows, slabs, align), plain)
    # distinct (row, slab) pairs land on distinct bytes
    if rows:
        marks = np.arange(rows * slabs, dtype=np.int64).reshape(rows, slabs)
        for v in (marks % 251, marks // 251 % 251):
            back = M.act_sf_untile(M.act_sf_tile(v.astype(np.uint8), align), rows, slabs, align)
            assert np.array_equal(back, v.astype(np.uint8))


def test_act_sf_layout_formula(M):
    # the byte of (r, s) sits where the header's formula says (spot checks, block rows 16 and 128)
    for align, rows, slabs in ((16, 70, 9), (256, 300, 6)):
        bt = M.act_sf_block_rows(align)
        nb = (rows + bt - 1) // bt + 1
        cb = 256 if bt == 16 else 512
        plain = np.zeros((rows, slabs), np.uint8)
        for r, s in ((0, 0), (rows - 1, slabs - 1), (17, 5), (rows // 2, 3)):
            plain[:] = 0
            plain[r, s] = 200
            tiled = M.act_sf_tile(plain, align)
            off = ((s // 4) * nb + r // bt) * cb + ((r % bt) % 32) * 16 + ((r % bt) // 32) * 4 + s % 4
            assert tiled[off] == 200


def test_invalid_arguments_are_rejected(M):
    L = M.lib()
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: validation fails first
    ws = ctypes.c_void_p(0x20000)
    # H not a multiple of 128
    assert L.moe_route(fake, fake, None, None, 8, 100, 16, 2, 0, 1, None, fake, fake, None, None, ws, 1 << 20,
                       None) == M.ERR_INVALID_ARG
    # K > E
    assert L.moe_route(fake, fake, None, None, 8, 128, 4, 5, 0, 1, None, fake, fake, None, None, ws, 1 << 20,
                       None) == M.ERR_INVALID_ARG
    # bad score function
    assert L.moe_route(fake, fake, None, None, 8, 128, 16, 2, 9, 1, None, fake, fake, None, None, ws, 1 << 20,
                       None) == M.ERR_INVALID_ARG
    # workspace too small
    assert L.moe_route(fake, fake, None, None, 8, 128, 16, 2, 0, 1, None, fake, fake, None, None, ws, 16,
                       None) == M.ERR_WORKSPACE
    # align not a power of two
    assert L.moe_permute(fake, 8, 2, 16, 3, fake, fake, fake, fake, None, None, None, 0, None, None, ws, 4096,
                         None) == M.ERR_INVALID_ARG
    # only some of the optional row-copy buffers
    assert L.moe_permute(fake, 8, 2, 16, 16, fake, fake, fake, fake, None, fake, None, 128, None, None, ws, 4096,
                         None) == M.ERR_INVALID_ARG
    # unsupported number of experts for the permute kernel
    assert L.moe_permute(fake, 8, 2, 4096, 16, fake, fake, fake, fake, None, None, None, 0, None, None, ws, 4096,
                         None) == M.ERR_UNSUPPORTED
    w = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 512, 2)
    # misaligned weight pointer
    wbad = M._Weight(0x10010, None, M.W_MXFP4, 16, 512, 512, 2)
    assert L.moe_grouped_gemm_l1_swiglu(fake, fake, 1, None, fake, fake, 8, 2, 512, 256, 16, 16, wbad, fake, fake, ws,
                                        4096, None) == M.ERR_INVALID_ARG
    # W13 must be packed with pair = 2 and the matching shape
    wpair = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 512, 1)
    assert L.moe_grouped_gemm_l1_swiglu(fake, fake, 1, None, fake, fake, 8, 2, 512, 256, 16, 16, wpair, fake, fake, ws,
                                        4096, None) == M.ERR_INVALID_ARG
    # token-order input (a_is_permuted = 0) needs sorted_token_ids
    assert L.moe_grouped_gemm_l1_swiglu(fake, fake, 0, None, fake, fake, 8, 2, 512, 256, 16, 16, w, fake, fake, ws,
                                        4096, None) == M.ERR_INVALID_ARG
    assert L.moe_grouped_ffn(fake, fake, 0, None, fake, fake, 8, 2, 512, 256, 16, 16, w, w, fake, fake, fake, ws,
                             4096, None) == M.ERR_INVALID_ARG
    # scales without rows is a valid permute mode; rows without scales is not
    assert L.moe_permute(fake, 8, 2, 16, 16, fake, fake, fake, fake, None, fake, None, 128, fake, None, ws, 4096,
                         None) == M.ERR_INVALID_ARG
    # NVFP4 needs a tensor scale pointer
    wnv = M._Weight(0x10000, None, M.W_NVFP4, 16, 512, 256, 1)
    assert L.moe_grouped_gemm_l2(fake, fake, fake, fake, 8, 2, 512, 256, 16, 16, wnv, fake, ws, 4096,
                                 None) == M.ERR_INVALID_ARG
    # forward with a workspace smaller than moe_workspace_size
    w2 = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 256, 1)
    assert L.moe_forward(fake, fake, None, None, 8, 512, 256, 16, 4, 16, 0, 1, w, w2, fake, None, None, None, None,
                         None, None, ws, 1024, None) == M.ERR_WORKSPACE
    # unpermute-reduce with H not a multiple of 8
    assert L.moe_unpermute_reduce(fake, fake, fake, 2, 2, 12, fake, None) == M.ERR_INVALID_ARG
    assert M.status_str(M.ERR_TIMEOUT) == "device wait timed out"


def test_single_launch_refusals_on_the_host(M):
    # moe_forward_single_launch validates as moe_forward does, then refuses what its one launch does
    # not cover (more than 16 tokens, more than 128 (token, slot) pairs, GEMM blocks above 16 rows,
    # NVFP4) before any device work
    L = M.lib()
    fake = ctypes.c_void_p(0x10000)     # never dereferenced
    ws = ctypes.c_void_p(0x20000)
    big = 1 << 40

    def call(T, K, align, w13, w2, ws_bytes):
        return L.moe_forward_single_launch(fake, fake, None, None, T, 512, 256, 16, K, align, 0, 1, w13, w2, fake,
                                           None, None, None, None, None, None, ws, ws_bytes, None)

    w13 = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 512, 2)
    w2 = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 256, 1)
    assert call(8, 4, 16, w13, w2, 1024) == M.ERR_WORKSPACE
    assert call(17, 4, 16, w13, w2, big) == M.ERR_UNSUPPORTED
    assert call(16, 9, 16, w13, w2, big) == M.ERR_UNSUPPORTED
    assert call(8, 4, 32, w13, w2, big) == M.ERR_UNSUPPORTED
    n13 = M._Weight(0x10000, 0x30000, M.W_NVFP4, 16, 512, 512, 2)
    n2 = M._Weight(0x10000, 0x30000, M.W_NVFP4, 16, 512, 256, 1)
    assert call(8, 4, 16, n13, n2, big) == M.ERR_UNSUPPORTED
    assert call(8, 4, 16, w13, M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 256, 2), big) == M.ERR_INVALID_ARG


def test_product_path_does_not_touch_the_oracle():
    # the library and its binding never import, load or call the oracle
    pkg = os.path.join(ROOT, "moe_expert_ffn_sqrt_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"(import|from)\s+oracle|oracle/", src), f


def test_variant_entry_points_reject_invalid_arguments(M):
    L = M.lib()
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: validation fails first
    ws = ctypes.c_void_p(0x20000)
    n = ctypes.c_size_t(0)
    # BatchedExperts slot sizes: powers of two in [1, 4096]
    for bad in (0, 3, 8192):
        assert L.moe_workspace_size_batched(8, 512, 256, 16, 4, bad, ctypes.byref(n)) == M.ERR_INVALID_ARG
        assert L.moe_batched_align(8, 4, 16, bad) == 0
    assert L.moe_workspace_size_batched(8, 512, 256, 16, 4, 16, ctypes.byref(n)) == M.OK and n.value > 0
    # the row-block height: the slot below 16 rows, else 64 (128 once experts average > 64 tokens)
    assert [L.moe_batched_align(8, 4, 16, s) for s in (1, 8, 16, 32, 64, 128, 4096)] == [1, 8, 16, 32, 64, 64, 64]
    assert L.moe_batched_align(4096, 6, 256, 4096) == 128
    assert L.moe_permute_batched(fake, 8, 2, 16, 12, fake, fake, fake, fake, None, None, None, 0, None, None, ws,
                                 1 << 20, None) == M.ERR_INVALID_ARG
    w13 = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 512, 2)
    w2 = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 256, 1)
    # a slot smaller than the batch
    assert L.moe_forward_batched(fake, fake, None, None, 9, 512, 256, 16, 4, 8, 0, 1, w13, w2, fake, None, None, None,
                                 None, None, None, None, ws, 1 << 30, None) == M.ERR_INVALID_ARG
    # the tiny-batch path: at most 16 tokens and T*K <= E
    assert L.moe_forward_naive(fake, fake, None, None, 17, 512, 256, 1024, 4, 0, 1, w13, w2, fake, None, None, None,
                               None, None, None, ws, 1 << 30, None) == M.ERR_UNSUPPORTED
    assert L.moe_forward_naive(fake, fake, None, None, 5, 512, 256, 16, 4, 0, 1, w13, w2, fake, None, None, None,
                               None, None, None, ws, 1 << 30, None) == M.ERR_UNSUPPORTED
    assert L.moe_route_naive(fake, fake, None, None, 5, 512, 16, 4, 0, 1, fake, fake, fake, fake, fake, fake, fake,
                             fake, ws, 1 << 20, None) == M.ERR_UNSUPPORTED
    # weighted L1 needs both the row ids and the weights
    assert L.moe_grouped_gemm_l1_swiglu_weighted(fake, fake, fake, fake, None, fake, 8, 2, 512, 256, 16, 16, w13,
                                                 fake, fake, ws, 1 << 20, None) == M.ERR_INVALID_ARG
    # failure-path self-test: workspace and mode checked on the host
    assert L.moe_selftest_wait_timeout(None, 256, 0, None) == M.ERR_INVALID_ARG
    assert L.moe_selftest_wait_timeout(ws, 128, 0, None) == M.ERR_INVALID_ARG
    assert L.moe_selftest_wait_timeout(ws, 256, 2, None) == M.ERR_INVALID_ARG


def test_int8_entry_points_reject_invalid_arguments(M):
    L = M.lib()
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: validation fails first
    ws = ctypes.c_void_p(0x20000)
    n = ctypes.c_size_t(0)
    # the packed INT8 stream: 256-row tiles x 64-deep slabs of one byte per code (W2 [2, 384, 256] pads a half tile)
    assert M.weight_packed_bytes("int8", 2, 512, 512, 2) == 2 * 512 * 512
    assert M.weight_packed_bytes("int8", 2, 384, 256, 1) == 2 * 2 * 4 * 256 * 64
    assert L.moe_workspace_size_i8(8, 512, 256, 16, 4, 16, ctypes.byref(n)) == M.OK
    assert n.value > M.workspace_size(8, 512, 256, 16, 4, 16)
    i13 = M._Weight(0x10000, 0x30000, M.W_INT8, 16, 512, 512, 2)
    i2 = M._Weight(0x10000, 0x30000, M.W_INT8, 16, 512, 256, 1)
    f13 = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 512, 2)
    f2 = M._Weight(0x10000, None, M.W_MXFP4, 16, 512, 256, 1)
    big = 1 << 30
    # INT8 weights only through the INT8 calls, FP4 weights never through them
    assert L.moe_forward(fake, fake, None, None, 8, 512, 256, 16, 4, 16, 0, 1, i13, i2, fake, None, None, None, None,
                         None, None, ws, big, None) == M.ERR_INVALID_ARG
    assert L.moe_forward_i8(fake, fake, None, None, 8, 512, 256, 16, 4, 16, 0, 1, f13, f2, fake, None, None, None,
                            None, None, None, ws, big, None) == M.ERR_INVALID_ARG
    # channel scales are required (and 16-byte aligned)
    for bad in (M._Weight(0x10000, None, M.W_INT8, 16, 512, 512, 2), M._Weight(0x10000, 0x30004, M.W_INT8, 16, 512, 512, 2)):
        assert L.moe_grouped_gemm_l1_swiglu_i8(fake, fake, fake, fake, fake, 8, 4, 512, 256, 16, 16, bad, fake, fake,
                                               ws, big, None) == M.ERR_INVALID_ARG
    # L2 needs W2's shape ([E, H, I], pair 1)
    assert L.moe_grouped_gemm_l2_i8(fake, fake, fake, fake, 8, 4, 512, 256, 16, 16, i13, fake, ws, big,
                                    None) == M.ERR_INVALID_ARG
    # workspace smaller than moe_workspace_size_i8
    assert L.moe_forward_i8(fake, fake, None, None, 8, 512, 256, 16, 4, 16, 0, 1, i13, i2, fake, None, None, None,
                            None, None, None, ws, n.value - 1, None) == M.ERR_WORKSPACE
    # per-row quantisation: columns a multiple of 128, 16-byte aligned buffers
    assert L.moe_act_quant_i8(fake, 4, 100, fake, fake, None) == M.ERR_INVALID_ARG
    assert L.moe_act_quant_i8(ctypes.c_void_p(0x10008), 4, 128, fake, fake, None) == M.ERR_INVALID_ARG
    # packing INT8 codes wants a 16-byte aligned source
    assert L.moe_pack_weights(M.W_INT8, ctypes.c_void_p(0x10004), None, 2, 512, 512, 2, fake, None) == M.ERR_INVALID_ARG
    # the INT8 BatchedExperts layout: power-of-two slots, no smaller than the batch
    for bad in (0, 3, 8192):
        assert L.moe_workspace_size_batched_i8(8, 512, 256, 16, 4, bad, ctypes.byref(n)) == M.ERR_INVALID_ARG
    assert L.moe_workspace_size_batched_i8(8, 512, 256, 16, 4, 16, ctypes.byref(n)) == M.OK and n.value > 0
    assert L.moe_forward_batched_i8(fake, fake, None, None, 9, 512, 256, 16, 4, 8, 0, 1, i13, i2, fake, None, None,
                                    None, None, None, None, None, ws, big, None) == M.ERR_INVALID_ARG
    assert L.moe_forward_batched_i8(fake, fake, None, None, 8, 512, 256, 16, 4, 16, 0, 1, f13, f2, fake, None, None,
                                    None, None, None, None, None, ws, big, None) == M.ERR_INVALID_ARG
