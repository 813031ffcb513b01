"""The C ABI library builds, loads, exports every declared symbol and rejects
bad arguments on the host before any launch (CPU only: no compute call
reaches a GPU here)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bl_attn.h")


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_fwd_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH) or not build.up_to_date():
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build libbl_attn.so")
        build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bl_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    from block_sparse_attention_fwd_gb300 import _lib
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _shape(**kw):
    from block_sparse_attention_fwd_gb300 import _lib
    a = dict(B=1, n=256, H=2, Hk=1, d=64, block_q=64, block_k=64)
    a.update(kw)
    return _lib.make_shape(**a)


def test_size_queries(lib):
    from block_sparse_attention_fwd_gb300 import _lib
    s = _shape(n=1000, block_q=128, block_k=64)
    assert _lib.tile_stats_elems(s) == 1 * 2 * 16 * (8 * 128)
    ws = _lib.bwd_workspace_bytes(s)
    assert ws >= 2 * 1000 * 4 + 1000 * 2 * 64 * 4 + 4
    assert _lib.tile_stats_elems(_shape(d=96)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(H=3, Hk=2), 1), (dict(n=0), 1), (dict(block_k=32), 2),
    (dict(B=0), 1)])
def test_fwd_rejects_bad_shapes_without_launching(lib, kw, code):
    s = _shape(**kw)
    fake = ctypes.c_void_p(0x10000)
    r = lib.bl_attn_fwd(ctypes.byref(s), fake, fake, fake, 0.125, fake, fake, None, None)
    assert r == code


def test_fwd_rejects_bad_pointers_and_scale(lib):
    s = _shape()
    ok = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    assert lib.bl_attn_fwd(ctypes.byref(s), None, ok, ok, 0.1, ok, ok, None, None) == 1
    assert lib.bl_attn_fwd(ctypes.byref(s), odd, ok, ok, 0.1, ok, ok, None, None) == 1
    assert lib.bl_attn_fwd(ctypes.byref(s), ok, ok, ok, 0.0, ok, ok, None, None) == 1
    assert lib.bl_attn_fwd(ctypes.byref(s), ok, ok, ok, float("nan"), ok, ok, None, None) == 1


def test_mask_rejects_bad_negl_prob(lib):
    from block_sparse_attention_fwd_gb300 import _lib
    s = _shape()
    ok = ctypes.c_void_p(0x10000)
    L = _lib.Lists(ok, ok, ok, ok, ok, None)
    for p in (-0.1, 1.0, 1.5, float("nan")):
        assert lib.bl_mask_from_stats(ctypes.byref(s), ok, ok, p, ctypes.byref(L), None) == 1
    L2 = _lib.Lists(ok, None, ok, ok, ok, None)
    assert lib.bl_mask_from_stats(ctypes.byref(s), ok, ok, 0.05, ctypes.byref(L2), None) == 1


def test_bwd_rejects_small_workspace(lib):
    from block_sparse_attention_fwd_gb300 import _lib
    s = _shape()
    ok = ctypes.c_void_p(0x10000)
    need = _lib.bwd_workspace_bytes(s)
    r = lib.bl_attn_bwd(ctypes.byref(s), ok, ok, ok, ok, ok, ok, 0.125, None, ok, ok, ok,
                        ok, need - 1, None)
    assert r == 4
    r = lib.bl_attn_bwd(ctypes.byref(s), ok, ok, ok, ok, ok, ok, 0.125, None, ok, ok, ok,
                        None, need, None)
    assert r == 4


def test_status_strings(lib):
    for c in range(7):
        assert lib.bl_status_string(c)


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "block_sparse_attention_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", src, re.M), f


def test_combine_rejects_bad_arguments(lib):
    ok = ctypes.c_void_p(0x10000)
    assert lib.bl_lse_combine(0, 1, 8, 1, 64, ok, ok, ok, ok, None) == 1
    assert lib.bl_lse_combine(33, 1, 8, 1, 64, ok, ok, ok, ok, None) == 1
    assert lib.bl_lse_combine(2, 1, 8, 1, 96, ok, ok, ok, ok, None) == 2
    assert lib.bl_lse_combine(2, 1, 8, 1, 64, None, ok, ok, ok, None) == 1


@pytest.mark.parametrize("kw,code", [
    (dict(causal=0, window=64, block_q=128, block_k=128), 1),     # a window needs causal
    (dict(causal=2, block_q=128, block_k=128), 1),
    (dict(causal=1, window=-1, block_q=128, block_k=128), 1),
    (dict(causal=1), 2),                                           # 64 x 64 tiles
    (dict(causal=1, block_q=128, block_k=64), 2)])
def test_causal_shape_checks(lib, kw, code):
    s = _shape(**kw)
    fake = ctypes.c_void_p(0x10000)
    assert lib.bl_attn_fwd(ctypes.byref(s), fake, fake, fake, 0.125, fake, fake, None, None) == code


def test_grad_error_rejects_bad_arguments(lib):
    ok = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    assert lib.bl_grad_error(None, ok, 8, ok, None) == 1
    assert lib.bl_grad_error(ok, ok, 0, ok, None) == 1
    assert lib.bl_grad_error(odd, ok, 8, ok, None) == 1
    assert lib.bl_grad_error(ok, ok, 8, ctypes.c_void_p(0x10004), None) == 1


def _varlen(cu, **kw):
    from block_sparse_attention_fwd_gb300 import _lib
    a = dict(H=4, Hk=2, d=64, block_q=128, block_k=128, causal=0, window=0, streams=0)
    a.update(kw)
    arr = (ctypes.c_int32 * len(cu))(*cu)
    v = _lib.VarlenStruct(len(cu) - 1, arr, a["H"], a["Hk"], a["d"], a["block_q"],
                          a["block_k"], a["causal"], a["window"], a["streams"])
    return v, arr


@pytest.mark.parametrize("cu,bq,bk", [
    ([0, 1, 129, 257, 385, 1000, 1000, 1300], 128, 128),
    ([0, 0, 300, 301, 301, 700], 64, 128),
    ([0, 5000], 128, 64),
    ([0, 64, 128, 192, 250, 250, 320], 64, 64)])
def test_varlen_layout_matches_the_oracle_layout(lib, cu, bq, bk):
    from block_sparse_attention_fwd_gb300 import _lib
    from oracle import varlen as OV
    v, arr = _varlen(cu, block_q=bq, block_k=bk)
    sz = _lib.VarlenSizes()
    assert lib.bl_varlen_layout(ctypes.byref(v), ctypes.byref(sz)) == 0
    _, tot = OV.layout(cu, 4, bq, bk)
    assert (sz.total, sz.lse, sz.tile_stats, sz.mask, sz.kv_cnt, sz.q_idx, sz.q_cnt) == \
        (tot["total"], tot["lse"], tot["stats"], tot["mask"], tot["kv_cnt"], tot["q_idx"],
         tot["q_cnt"])
    # one launch group per run of equal non-zero lengths
    lens = [b - a for a, b in zip(cu[:-1], cu[1:]) if b > a]
    assert sz.groups == sum(1 for i, n in enumerate(lens) if i == 0 or lens[i - 1] != n)
    # every run has its own D [B,H,n] and dQ [B,n,H,d] fp32 areas and a status slot
    runs = []
    for i, n in enumerate(lens):
        if i and lens[i - 1] == n:
            runs[-1][0] += 1
        else:
            runs.append([1, n])
    def sub(b, n):   # 64-wide tiles: lists regrouped into 128 x 128 tiles (+ counts)
        if bq == 128 and bk == 128:
            return 0
        t = -(-n // 128)
        return -(-(b * 4 * t * (t + 1) * 4) // 256) * 256

    want = sum(-(-(b * 4 * n * 4) // 256) * 256 + b * n * 4 * 64 * 4 + sub(b, n)
               for b, n in runs)
    assert sz.bwd_workspace_bytes == want + 16 * len(runs)


@pytest.mark.parametrize("cu,kw,code", [
    ([1, 5], {}, 1),                    # cu[0] != 0
    ([0, 9, 4], {}, 1),                 # decreasing
    ([0, 0, 0], {}, 1),                 # no tokens
    ([0], {}, 1),                       # no sequence
    ([0, 100], dict(d=96), 2),
    ([0, 100], dict(H=3, Hk=2), 1),
    ([0, 100], dict(causal=1, block_q=64, block_k=64), 2),
    ([0, 100], dict(window=8), 1),
    ([0, 100], dict(streams=-1), 1),
    ([0, 100], dict(streams=9), 1)])
def test_varlen_rejects_bad_descriptions(lib, cu, kw, code):
    from block_sparse_attention_fwd_gb300 import _lib
    v, arr = _varlen(cu, **kw)
    sz = _lib.VarlenSizes()
    assert lib.bl_varlen_layout(ctypes.byref(v), ctypes.byref(sz)) == code
    ok = ctypes.c_void_p(0x10000)
    assert lib.bl_attn_fwd_varlen(ctypes.byref(v), ok, ok, ok, 0.1, ok, ok, None, None) == code
    L = _lib.Lists(ok, ok, ok, ok, ok, None)
    assert lib.bl_mask_from_stats_varlen(ctypes.byref(v), ok, ok, 0.05, ctypes.byref(L),
                                         None) == code
    assert lib.bl_attn_bwd_varlen(ctypes.byref(v), ok, ok, ok, ok, ok, ok, 0.1, None, ok, ok,
                                  ok, ok, 1 << 30, None) == code
    assert lib.bl_varlen_layout(None, ctypes.byref(sz)) == 1


def test_varlen_calls_reject_bad_arguments_without_launching(lib):
    from block_sparse_attention_fwd_gb300 import _lib
    v, arr = _varlen([0, 100, 356])
    sz = _lib.VarlenSizes()
    assert lib.bl_varlen_layout(ctypes.byref(v), ctypes.byref(sz)) == 0
    ok, odd, odd4 = (ctypes.c_void_p(x) for x in (0x10000, 0x10004, 0x10002))
    V = ctypes.byref(v)
    assert lib.bl_attn_fwd_varlen(V, odd, ok, ok, 0.1, ok, ok, None, None) == 1
    assert lib.bl_attn_fwd_varlen(V, ok, ok, ok, 0.1, ok, odd4, None, None) == 1   # lse: 4 bytes
    assert lib.bl_attn_fwd_varlen(V, ok, ok, ok, 0.0, ok, ok, None, None) == 1
    assert lib.bl_attn_fwd_varlen(V, ok, ok, ok, 0.1, ok, ok, odd, None) == 1
    L = _lib.Lists(ok, ok, ok, ok, ok, None)
    for p in (-0.1, 1.0, float("nan")):
        assert lib.bl_mask_from_stats_varlen(V, ok, ok, p, ctypes.byref(L), None) == 1
    need = sz.bwd_workspace_bytes
    assert lib.bl_attn_bwd_varlen(V, ok, ok, ok, ok, ok, ok, 0.1, None, ok, ok, ok, ok,
                                  need - 1, None) == 4
    assert lib.bl_attn_bwd_varlen(V, ok, ok, ok, ok, ok, ok, 0.1, None, ok, ok, ok, None,
                                  need, None) == 4
    assert lib.bl_attn_bwd_varlen(V, ok, ok, ok, ok, ok, odd4, 0.1, None, ok, ok, ok, ok,
                                  need, None) == 1
    assert lib.bl_varlen_bwd_check_status(V, None, None) == 4


def test_varlen_long_sequence_limit_is_the_mask_passs_only(lib):
    from block_sparse_attention_fwd_gb300 import _lib
    v, arr = _varlen([0, 1000, 300000])           # T_c = 2336 > 2048 for the second
    sz = _lib.VarlenSizes()
    assert lib.bl_varlen_layout(ctypes.byref(v), ctypes.byref(sz)) == 0
    ok = ctypes.c_void_p(0x10000)
    L = _lib.Lists(ok, ok, ok, ok, ok, None)
    assert lib.bl_mask_from_stats_varlen(ctypes.byref(v), ok, ok, 0.05, ctypes.byref(L),
                                         None) == 2


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "bl_attn.h"

int main(void) {
  bl_shape s, s2;
  int32_t cu[4] = {0, 100, 100, 356};
  bl_varlen v;
  bl_varlen_sizes z;
  bl_status st;
  memset(&s, 0, sizeof s);
  s.B = 1; s.n = 1000; s.H = 2; s.Hk = 1; s.d = 64; s.block_q = 128; s.block_k = 64;
  printf("%zu %zu\n", bl_tile_stats_elems(&s), bl_bwd_workspace_bytes(&s));
  memset(&v, 0, sizeof v);
  v.nseq = 3; v.cu_seqlens = cu; v.H = 4; v.Hk = 2; v.d = 64; v.block_q = 128; v.block_k = 128;
  st = bl_varlen_layout(&v, &z);
  printf("%d %zu %zu %zu %zu %zu %zu %zu %zu %d\n", (int)st, z.total, z.lse, z.tile_stats, z.mask,
         z.kv_cnt, z.q_idx, z.q_cnt, z.bwd_workspace_bytes, z.groups);
  printf("%d\n", (int)bl_attn_fwd(&s, NULL, NULL, NULL, 0.125f, NULL, NULL, NULL, NULL));
  printf("%s\n", bl_status_string(BL_ERR_UNSUPPORTED));
  /* a kv-head slice view: strides of the full tensor; a last stride of 2 is refused */
  s2 = s;
  s2.q_strides[0] = 1000 * 8 * 64; s2.q_strides[1] = 8 * 64; s2.q_strides[2] = 64;
  s2.q_strides[3] = 1;
  printf("%zu", bl_tile_stats_elems(&s2));
  s2.q_strides[3] = 2;
  printf(" %zu\n", bl_tile_stats_elems(&s2));
  return 0;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    """The header compiles as C99 with warnings as errors, and a C program
    linked against the library gets the same sizes as the Python binding
    (host-side calls only: nothing reaches a GPU)."""
    import subprocess
    from block_sparse_attention_fwd_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(_lib.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-lbl_attn", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.strip().splitlines()
    s = _shape(n=1000, H=2, Hk=1, d=64, block_q=128, block_k=64)
    assert lines[0].split() == [str(_lib.tile_stats_elems(s)), str(_lib.bwd_workspace_bytes(s))]
    vl = _lib.Varlen([0, 100, 100, 356], 4, 2, 64, 128, 128)
    z = vl.sizes
    want = [0, z["total"], z["lse"], z["tile_stats"], z["mask"], z["kv_cnt"], z["q_idx"],
            z["q_cnt"], z["bwd_workspace_bytes"], z["groups"]]
    assert [int(x) for x in lines[1].split()] == want
    assert want[1:4] == [356, 4 * 356, 4 * 1 * 128 + 4 * 2 * 256] and want[-1] == 2
    assert lines[2] == "1"                           # BL_ERR_INVALID_ARG before any launch
    assert lines[3] == "unsupported configuration"
    assert lines[4].split() == [lines[0].split()[0], "0"]


def test_varlen_splits_runs_longer_than_the_grid_limit(lib):
    """70000 sequences of one token: a launch group holds at most 65535
    sequences (the grid's batch dimension), so the run splits in two; the
    sizes are still the sum over sequences."""
    from block_sparse_attention_fwd_gb300 import _lib
    cu = list(range(70001))
    v, arr = _varlen(cu, H=2, Hk=1, d=64, block_q=64, block_k=64)
    sz = _lib.VarlenSizes()
    assert lib.bl_varlen_layout(ctypes.byref(v), ctypes.byref(sz)) == 0
    assert sz.groups == 2
    assert (sz.total, sz.lse, sz.tile_stats, sz.mask, sz.kv_cnt) == \
        (70000, 2 * 70000, 2 * 64 * 70000, 2 * 70000, 2 * 70000)
    # one D area (256-byte rounded), one dQ area and (64-wide tiles) one area of
    # regrouped lists per group, one 16-byte slot each
    want = sum(-(-(b * 2 * 4) // 256) * 256 + b * 2 * 64 * 4 + -(-(b * 2 * 1 * 2 * 4) // 256) * 256
               for b in (65535, 4465)) + 2 * 16
    assert sz.bwd_workspace_bytes == want


def test_list_sizes_match_the_documented_layout(lib):
    from block_sparse_attention_fwd_gb300 import _lib
    s = _shape(B=2, n=1000, H=4, Hk=2, d=64, block_q=128, block_k=64)   # T_r 8, T_c 16
    m, kv, kc, qi, qc, total = _lib.lists_elems(s)
    assert (m, kv, kc, qi, qc) == (2 * 4 * 8 * 16, 2 * 4 * 8 * 16, 2 * 4 * 8, 2 * 4 * 16 * 8,
                                   2 * 4 * 16)
    assert total == m + 4 * (kv + kc + qi + qc)
    got = _lib.alloc_lists(s, "cpu")                       # the binding allocates the same sizes
    assert [got[k].numel() for k in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt")] == \
        [m, kv, kc, qi, qc]
    out = (ctypes.c_size_t * 5)()
    assert lib.bl_lists_elems(ctypes.byref(_shape(d=96)), out) == 0
    assert lib.bl_lists_elems(ctypes.byref(s), None) == 0


def test_varlen_layout_matches_the_oracle_on_random_batches(lib):
    """200 seeded random packings (empty sequences, runs of equal lengths,
    both tile sizes): the library's sizes equal the oracle's layout and its
    launch groups are the runs of equal non-zero lengths."""
    import numpy as np
    from block_sparse_attention_fwd_gb300 import _lib
    from oracle import varlen as OV
    rng = np.random.default_rng(11)
    for _ in range(200):
        nseq = int(rng.integers(1, 12))
        pool = rng.integers(0, 700, size=3)
        lens = [int(pool[rng.integers(0, 3)]) if rng.random() < 0.5 else int(rng.integers(0, 700))
                for _ in range(nseq)]
        lens = [0 if rng.random() < 0.15 else n for n in lens]      # empty sequences
        if sum(lens) == 0:
            lens[0] = 1
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(int).tolist()
        bq, bk = (int(x) for x in rng.choice([64, 128], size=2))
        causal = int(bq == 128 and bk == 128 and rng.random() < 0.5)
        v, arr = _varlen(cu, H=2, Hk=1, d=64, block_q=bq, block_k=bk, causal=causal)
        sz = _lib.VarlenSizes()
        assert lib.bl_varlen_layout(ctypes.byref(v), ctypes.byref(sz)) == 0
        _, tot = OV.layout(cu, 2, bq, bk)
        assert (sz.total, sz.lse, sz.tile_stats, sz.mask, sz.kv_cnt, sz.q_idx, sz.q_cnt) == \
            (tot["total"], tot["lse"], tot["stats"], tot["mask"], tot["kv_cnt"], tot["q_idx"],
             tot["q_cnt"]), (cu, bq, bk)
        # a group is a run of consecutive sequences of one non-zero length (an
        # empty sequence ends a run)
        assert sz.groups == sum(1 for i, n in enumerate(lens) if n and (i == 0 or lens[i - 1] != n))


def test_strided_shapes_are_validated_on_the_host(lib):
    """bl_shape strides: zero means contiguous; otherwise the dim stride is 1,
    the others positive multiples of 8 elements, the head stride at least d."""
    from block_sparse_attention_fwd_gb300 import _lib
    base = _lib.make_shape(1, 1000, 4, 2, 64, 128, 128)
    want = _lib.tile_stats_elems(base)

    def with_q(st):
        s = _lib.Shape.from_buffer_copy(base)
        for i, x in enumerate(st):
            s.q_strides[i] = x
        return s

    # a view of heads 4..7 of an [1, 1000, 16, 64] tensor
    assert _lib.tile_stats_elems(with_q((1000 * 16 * 64, 16 * 64, 64, 1))) == want
    for bad in ((1000 * 16 * 64, 16 * 64, 64, 2),     # dim stride must be 1
                (1000 * 16 * 64, 16 * 64 + 4, 64, 1),  # not a multiple of 8
                (1000 * 16 * 64, 16 * 64, 32, 1),      # heads overlap
                (0, 16 * 64, 64, 1)):                  # non-positive
        assert _lib.tile_stats_elems(with_q(bad)) == 0


def test_wait_limit_knob_clamps_and_restores(lib):
    """bl_set_wait_limit (host only): [0, 2) s is taken as given, anything else
    restores 2 s; each call returns the previous limit."""
    from block_sparse_attention_fwd_gb300 import _lib
    assert _lib.set_wait_limit(0.25) == pytest.approx(2.0)
    assert _lib.set_wait_limit(5.0) == pytest.approx(0.25)
    assert _lib.set_wait_limit(0.0) == pytest.approx(2.0)
    assert _lib.set_wait_limit(-1.0) == 0.0
    assert _lib.set_wait_limit(-1.0) == pytest.approx(2.0)
