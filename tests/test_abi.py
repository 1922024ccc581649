"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and its host-side logic (RoPE table, pool size, planner, argument
validation) behaves as specified.  Validation failures return before any CUDA
call, so they are testable here."""
import ctypes
import json
import math
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pkv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for n in ("pkv_append_rope", "pkv_decode_attention", "pkv_prefill_attention_ragged",
              "pkv_merge_states", "pkv_gather_kv", "pkv_decode_workspace_size",
              "pkv_prefill_workspace_size", "pkv_rope_cos_sin_table", "pkv_last_error",
              "pkv_decode_plan", "pkv_cache_bytes", "pkv_device_errors"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(pkv.library_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_rope_table_equals_oracle_bit_for_bit(lib):
    for theta, dim, n in ((1e6, 128, 4096), (1e4, 64, 1000), (5e5, 128, 100)):
        a = pkv.pkv_rope_cos_sin_table(theta, dim, n)
        b = oracle.rope_table(theta, dim, n)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_pool_bytes_match_the_printed_kv_pool_size(lib):
    g = json.load(open(os.path.join(GOLDEN, "kv_pool_bytes.json")))
    for dtype, printed in ((pkv.KV_BF16, g["bf16_gb_printed"]), (pkv.KV_FP8_E4M3,
                                                                  g["fp8_gb_printed"])):
        d = pkv.make_desc(num_q_heads=16, num_kv_heads=g["num_kv_heads"], head_dim=g["head_dim"],
                          num_blocks=g["num_blocks"], max_blocks_per_seq=1, kv_dtype=dtype,
                          block_size=g["block_size"])
        total = pkv.pkv_cache_bytes(d) * 2 * g["num_layers"]  # K and V, every layer
        assert abs(total / 1e9 - printed) <= g["printed_precision_gb"]


def _desc(**kw):
    base = dict(num_q_heads=16, num_kv_heads=2, head_dim=128, num_blocks=1000,
                max_blocks_per_seq=256)
    base.update(kw)
    return pkv.make_desc(**base)


def test_invalid_arguments_return_status_before_any_device_work(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: validation fails first
    cases = [
        (None, pkv.PkvError, 1),
    ]
    # null desc
    st = lib.pkv_decode_attention(None, fake, fake, fake, None, None, fake, fake, 1, 10, 0.1, -1,
                                  None, 0, fake, None, None, 0, None)
    assert st == 1 and "desc" in pkv.pkv_last_error()
    bad = [
        (_desc(num_q_heads=15), 1, "multiple"),
        (_desc(head_dim=96), 2, "head_dim"),
        (_desc(num_q_heads=64, num_kv_heads=2), 2, "group"),
        (_desc(block_size=32), 2, "block_size"),
        (_desc(kv_dtype=7), 2, "kv_dtype"),
        (_desc(num_blocks=0), 1, "num_blocks"),
        (_desc(flags=0x4), 1, "flags"),
    ]
    for d, code, word in bad:
        st = lib.pkv_decode_attention(ctypes.byref(d), fake, fake, fake, None, None, fake, fake, 1,
                                      10, 0.1, -1, None, 0, fake, None, None, 0, None)
        assert st == code, (word, st)
        assert word in pkv.pkv_last_error()
    d = _desc()
    # context longer than the table can hold
    st = lib.pkv_decode_attention(ctypes.byref(d), fake, fake, fake, None, None, fake, fake, 1,
                                  256 * 16 + 1, 0.1, -1, None, 0, fake, None, None, 0, None)
    assert st == 1 and "max_context_len" in pkv.pkv_last_error()
    # e4m3 without scales
    d8 = _desc(kv_dtype=pkv.KV_FP8_E4M3)
    st = lib.pkv_decode_attention(ctypes.byref(d8), fake, fake, fake, None, None, fake, fake, 1,
                                  10, 0.1, -1, None, 0, fake, None, None, 0, None)
    assert st == 1 and "scale" in pkv.pkv_last_error()
    # null pointers
    st = lib.pkv_decode_attention(ctypes.byref(d), None, fake, fake, None, None, fake, fake, 1,
                                  10, 0.1, -1, None, 0, fake, None, None, 0, None)
    assert st == 1
    # misaligned q
    st = lib.pkv_decode_attention(ctypes.byref(d), P(0x10002), fake, fake, None, None, fake, fake,
                                  1, 10, 0.1, -1, None, 0, fake, None, None, 0, None)
    assert st == 1 and "aligned" in pkv.pkv_last_error()
    # bad sm_scale
    st = lib.pkv_decode_attention(ctypes.byref(d), fake, fake, fake, None, None, fake, fake, 1,
                                  10, float("nan"), -1, None, 0, fake, None, None, 0, None)
    assert st == 1
    # zero sequences: a no-op, OK
    st = lib.pkv_decode_attention(ctypes.byref(d), None, None, None, None, None, None, None, 0,
                                  10, 0.1, -1, None, 0, None, None, None, 0, None)
    assert st == 0
    # prefill: e4m3 pools need their scales; kv_len < q_len rejected
    st = lib.pkv_prefill_attention_ragged(ctypes.byref(d8), fake, fake, fake, fake, None, None,
                                          fake, fake, 1, 4, None, None, 0.1, 1, -1, fake, None,
                                          None, 0, None)
    assert st == 1 and "scale" in pkv.pkv_last_error()
    qo = np.array([0, 4], np.int32)
    kl = np.array([3], np.int32)
    st = lib.pkv_prefill_attention_ragged(ctypes.byref(d), fake, fake, fake, fake, None, None,
                                          fake, fake, 1, 4, qo.ctypes.data_as(P),
                                          kl.ctypes.data_as(P), 0.1, 1, -1, fake, None, None, 0,
                                          None)
    assert st == 1 and "kv_len" in pkv.pkv_last_error()
    # append and merge
    st = lib.pkv_append_rope(ctypes.byref(d), None, fake, None, None, fake, 1, fake, fake, 1, fake,
                             fake, None, None, 0, None)
    assert st == 1
    st = lib.pkv_merge_states(None, None, 2, 4, 4, 64, fake, None, None)
    assert st == 1
    st = lib.pkv_rope_cos_sin_table(1e4, 63, 10, fake)
    assert st == 1
    # ring cache: bounded by the table row, needs a window it can hold; prefill refuses it
    st = lib.pkv_decode_attention(ctypes.byref(_desc(max_blocks_per_seq=8, ring_blocks=9)), fake, fake,
                                  fake, None, None, fake, fake, 1, 10, 0.1, 128, None, 0, fake, None,
                                  None, 0, None)
    assert st == 1 and "ring_blocks" in pkv.pkv_last_error()
    dr = _desc(ring_blocks=9)
    for window in (-1, 0, 145):
        st = lib.pkv_decode_attention(ctypes.byref(dr), fake, fake, fake, None, None, fake, fake, 1,
                                      100000, 0.1, window, None, 0, fake, None, None, 0, None)
        assert st == 1 and "window" in pkv.pkv_last_error(), window
    st = lib.pkv_prefill_attention_ragged(ctypes.byref(dr), fake, fake, fake, fake, None, None,
                                          fake, fake, 1, 4, None, None, 0.1, 1, -1, fake, None,
                                          None, 0, None)
    assert st == 2 and "ring" in pkv.pkv_last_error()


def test_decode_step_validates_its_new_token_arguments(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    d = _desc()

    def step(k_new, v_new, cos_sin, max_pos, max_ctx=100):
        return lib.pkv_decode_step(ctypes.byref(d), fake, k_new, v_new, cos_sin, max_pos, fake, fake,
                                   None, None, fake, fake, 1, max_ctx, 0.1, -1, None, 0, fake, None,
                                   None, 0, None)

    assert step(None, fake, None, 0) == 1 and "k_new" in pkv.pkv_last_error()
    assert step(fake, None, None, 0) == 1 and "v_new" in pkv.pkv_last_error()
    assert step(P(0x10008), fake, None, 0) == 1 and "aligned" in pkv.pkv_last_error()
    # the table must cover the new token's position max_context_len - 1
    assert step(fake, fake, fake, 99) == 1 and "rope_max_pos" in pkv.pkv_last_error()
    # the shared checks of decode still apply
    assert step(fake, fake, fake, 4097, max_ctx=256 * 16 + 1) == 1
    assert "max_context_len" in pkv.pkv_last_error()


def test_bound_decode_step_reports_argument_errors_when_called(lib):
    import torch
    d = _desc()
    q = torch.zeros((2, 16, 128), dtype=torch.bfloat16)
    t = torch.zeros((2, 256), dtype=torch.int32)
    l = torch.zeros(2, dtype=torch.int32)
    call = pkv.bind_decode_step(d, q, None, q, q, q, t, l, 100, 0.1, q, stream=0)
    with pytest.raises(pkv.PkvError, match="k_new"):
        call()


def test_planner_fills_the_gpu_and_respects_limits(lib):
    sms = 152
    # (Hq, Hkv, D, dtype, B, max_ctx, window)
    shapes = [(8, 2, 64, 0, 4, 255, -1), (16, 2, 128, 0, 64, 4096, -1),
              (32, 8, 128, 0, 256, 768, -1), (32, 8, 128, 0, 120, 32768, -1),
              (64, 8, 64, 1, 128, 16384, -1), (64, 8, 64, 1, 128, 16384, 128),
              (16, 2, 128, 0, 1, 1 << 19, -1)]
    for hq, hkv, d, dt, B, ctx, win in shapes:
        desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=10,
                             max_blocks_per_seq=(ctx + 15) // 16, kv_dtype=dt)
        chunk, splits = pkv.pkv_decode_plan(desc, B, ctx, win, sms)
        vis_blocks = (ctx + 15) // 16 if win <= 0 else min((ctx + 15) // 16, (win + 14) // 16 + 1)
        assert 1 <= chunk <= 256
        assert splits == math.ceil(vis_blocks / chunk) and splits <= 512
        if B * hkv * vis_blocks >= 16 * sms * 8:
            # large batches: enough CTAs for several waves, none smaller than 16 blocks
            assert B * hkv * splits >= sms and chunk >= 16
    # a window never needs more blocks than it can touch
    desc = pkv.make_desc(num_q_heads=64, num_kv_heads=8, head_dim=64, num_blocks=10,
                         max_blocks_per_seq=1024, kv_dtype=1)
    assert pkv.pkv_decode_plan(desc, 128, 16384, 128, sms) == (9, 1)
    # chunks above 128 blocks only while the batch spans >= 8 waves with them: the
    # Llama-3-8B-shaped decode (120 x 8 pairs, up to 2048 blocks) takes 256-block
    # chunks; the FP8 layer (e4m3, one block id per lane) stays at 128
    d8b = pkv.make_desc(num_q_heads=32, num_kv_heads=8, head_dim=128, num_blocks=10, max_blocks_per_seq=2048)
    assert pkv.pkv_decode_plan(d8b, 120, 32768, -1, sms) == (256, 8)
    assert pkv.pkv_decode_plan(desc, 128, 16384, -1, sms) == (128, 8)
    # a small bf16 batch of the same length spans few waves: 128 at most
    chunk, _ = pkv.pkv_decode_plan(d8b, 8, 32768, -1, sms)
    assert chunk <= 128
    # contexts past 512 chunks of the longest a CTA takes (256 blocks bf16, 128 e4m3) are refused
    for dt, limit in ((0, 512 * 256), (1, 512 * 128)):
        dl = pkv.make_desc(num_q_heads=16, num_kv_heads=2, head_dim=128, num_blocks=10,
                           max_blocks_per_seq=limit + 1, kv_dtype=dt)
        assert pkv.pkv_decode_plan(dl, 1, limit * 16, -1, sms)[1] == 512
        with pytest.raises(pkv.PkvError):
            pkv.pkv_decode_plan(dl, 1, limit * 16 + 1, -1, sms)


def test_workspace_size_layout(lib):
    d = _desc()
    B, ctx = 10, 1000  # 63 blocks
    assert pkv.pkv_decode_workspace_size(d, B, ctx, -1, 64) == 0  # one split: none needed
    sz = pkv.pkv_decode_workspace_size(d, B, ctx, -1, 16)  # 4 splits
    pairs, G, D, S = B * 2, 8, 128, 4
    a256 = lambda x: (x + 255) // 256 * 256
    assert sz == a256(pairs * 4) + a256(pairs * S * G * 4) + a256(pairs * S * G * D * 4)
    assert pkv.pkv_decode_workspace_size(d, B, ctx, -1, 257) == 0  # chunk > 256 rejected
    # 250 blocks: chunks of 200 (bf16) or 128 (e4m3) give two; an e4m3 chunk above 128 is refused
    assert pkv.pkv_decode_workspace_size(d, 4, 4000, -1, 200) > 0
    d8 = _desc(num_q_heads=64, num_kv_heads=8, head_dim=64, kv_dtype=pkv.KV_FP8_E4M3)
    assert pkv.pkv_decode_workspace_size(d8, 4, 4000, -1, 128) > 0
    assert pkv.pkv_decode_workspace_size(d8, 4, 4000, -1, 129) == 0


def test_wait_timeout_hook_validates_its_arguments(lib):
    """The test hook is off by default and checks its arguments on the host."""
    with pytest.raises(pkv.PkvError):
        pkv.pkv_test_inject_wait_timeout(4, 1000)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_test_inject_wait_timeout(1, 0)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_test_inject_wait_timeout(1, 2000000)
    pkv.pkv_test_inject_wait_timeout(0)
