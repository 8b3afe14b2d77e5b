"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol that include/dsa_indexer.h declares, and rejects bad arguments on the
host before touching the device."""
import ctypes
import os
import re

import pytest

from infra_dsa_indexer_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa_indexer.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"IDX_API\s+[\w\s\*]+?\b(indexer_\w+)\s*\(", text)))


def test_header_declares_the_api():
    syms = declared_symbols()
    assert "indexer_logits" in syms and "indexer_get_last_error" in syms
    assert len(syms) >= 7


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        getattr(lib, name)


def test_binding_exposes_same_names():
    for name in declared_symbols():
        assert callable(getattr(binding, name)), name


def test_status_strings(lib):
    for st in range(0, 11):
        assert binding.indexer_status_string(st)
    assert "unknown" in binding.indexer_status_string(12345)
    assert binding.indexer_version() >= 100
    assert binding.indexer_launches_per_call(shp()) == 1
    assert binding.indexer_launches_per_call(shp(flags=1)) == 2
    assert binding.indexer_launches_per_call(shp(flags=1, S=16388)) == 2   # any S
    assert binding.indexer_launches_per_call(shp(fmt=2)) == 2              # MX: scale order
    assert binding.indexer_launches_per_call(shp(fmt=3, flags=1)) == 3


FAKE = ctypes.c_void_p(0x1000)      # never dereferenced: validation fails first


def call(lib, shape, **over):
    args = dict(q=FAKE, q_sf=None, k=FAKE, k_sf=None, k_scales=None, w=FAKE, ks=FAKE, ke=FAKE,
                sm_scale=ctypes.c_float(0.1), clean=1, out=FAKE)
    args.update(over)
    return lib.indexer_logits(args["q"], args["q_sf"], args["k"], args["k_sf"],
                              args["k_scales"], args["w"], args["ks"], args["ke"],
                              args["sm_scale"], args["clean"], args["out"],
                              ctypes.byref(shape), None)


def shp(**kw):
    base = dict(B=1, S=8, N=100, H=64, D=128, fmt=0, w_fmt=0, flags=0)
    base.update(kw)
    return binding.make_shape(**base)


@pytest.mark.parametrize("over,shape_kw,status", [
    (dict(q=None), {}, 1),
    (dict(out=None), {}, 1),
    ({}, dict(H=32), 2),
    ({}, dict(D=64), 2),
    ({}, dict(S=0), 2),
    ({}, dict(N=0), 2),
    ({}, dict(B=0), 2),
    ({}, dict(flags=4), 2),                               # unknown flag bit
    (dict(out=ctypes.c_void_p(0x1002)), {}, 4),           # FP32 out not 4-byte aligned
    (dict(out=ctypes.c_void_p(0x1001)), dict(flags=2), 4),  # BF16 out not 2-byte aligned
    ({}, dict(out_row_stride=50), 2),
    ({}, dict(fmt=7), 3),
    ({}, dict(w_fmt=3), 3),
    ({}, dict(fmt=2), 1),                                 # MX without scales
    (dict(q_sf=FAKE, k_sf=FAKE), dict(fmt=0), 3),         # scales for a plain format
    (dict(k_scales=FAKE), dict(fmt=0), 3),                # per-key scale only for E4M3
    (dict(q=ctypes.c_void_p(0x1004)), {}, 4),             # misaligned base
    ({}, dict(k_row_bytes=264), 4),                       # stride not a multiple of 16
    (dict(sm_scale=ctypes.c_float(float("inf"))), {}, 5),
    (dict(sm_scale=ctypes.c_float(float("nan"))), {}, 5),
])
def test_host_validation(lib, over, shape_kw, status):
    assert call(lib, shp(**shape_kw), **over) == status


@pytest.mark.parametrize("shape_kw,status", [(dict(H=32), 2), (dict(fmt=9), 3),
                                              (dict(out_row_stride=7), 2)])
def test_noalloc_entry_validates_like_indexer_logits(lib, shape_kw, status):
    args = (FAKE, None, FAKE, None, None, FAKE, FAKE, FAKE, ctypes.c_float(0.1), 1, FAKE)
    assert lib.indexer_logits_noalloc(*args, ctypes.byref(shp(**shape_kw)), None) == status
    assert lib.indexer_logits_noalloc(FAKE, None, None, None, None, FAKE, FAKE, FAKE,
                                      ctypes.c_float(0.1), 1, FAKE,
                                      ctypes.byref(shp()), None) == 1


def test_null_shape(lib):
    assert lib.indexer_logits(FAKE, None, FAKE, None, None, FAKE, FAKE, FAKE,
                              ctypes.c_float(1.0), 1, FAKE, None, None) == 1


def test_binding_raises_without_cuda_tensors(lib):
    import torch
    t = torch.zeros(4)
    with pytest.raises(ValueError):
        binding.indexer_logits(t, None, t, None, None, t, t, t, 1.0, True, t, shp())


def paged_call(lib, shape, paged, **over):
    args = dict(q=FAKE, q_sf=None, k=FAKE, k_sf=None, k_scales=None, w=FAKE, ks=FAKE, ke=FAKE,
                sm_scale=ctypes.c_float(0.1), clean=1, out=FAKE)
    args.update(over)
    return lib.indexer_paged_logits(args["q"], args["q_sf"], args["k"], args["k_sf"],
                                    args["k_scales"], args["w"], args["ks"], args["ke"],
                                    args["sm_scale"], args["clean"], args["out"],
                                    ctypes.byref(shape),
                                    ctypes.byref(paged) if paged is not None else None, None)


@pytest.mark.parametrize("paged_kw,shape_kw,status", [
    (None, {}, 1),                                            # no descriptor
    (dict(block_table=None), {}, 1),
    (dict(page_size=32), {}, 2),                              # not a multiple of 64
    (dict(page_size=0), {}, 2),
    (dict(table_stride=1), dict(N=100), 2),                   # needs ceil(100 / 64) = 2
    (dict(num_pages=0), {}, 2),
    (dict(reserved=1), {}, 2),
    ({}, dict(k_batch_bytes=4096), 2),                        # no batch stride in a cache
    (dict(num_pages=1 << 26), {}, 2),                         # rows beyond int32
])
def test_paged_host_validation(lib, paged_kw, shape_kw, status):
    pg = None
    if paged_kw is not None:
        base = dict(block_table=0x2000, table_stride=4, page_size=64, num_pages=8, reserved=0)
        base.update(paged_kw)
        pg = binding.idx_paged(ctypes.c_void_p(base["block_table"]), base["table_stride"],
                               base["page_size"], base["num_pages"], base["reserved"])
    assert paged_call(lib, shp(**shape_kw), pg) == status


@pytest.mark.parametrize("args,status", [
    (dict(logits=None), 1),
    (dict(idx=None), 1),
    (dict(rows=0), 2),
    (dict(N=0), 2),
    (dict(k=0), 2),
    (dict(row_stride=50), 2),                              # < N
    (dict(idx_stride=3), 2),                               # < k
    (dict(logits=ctypes.c_void_p(0x1002)), 4),             # FP32 not 4-byte aligned
    (dict(logits=ctypes.c_void_p(0x1001), bf16=1), 4),     # BF16 not 2-byte aligned
    (dict(idx=ctypes.c_void_p(0x1002)), 4),
])
def test_topk_host_validation(lib, args, status):
    a = dict(logits=FAKE, bf16=0, rows=4, N=100, row_stride=100, k=8, idx=FAKE, idx_stride=8)
    a.update(args)
    assert lib.indexer_topk(a["logits"], a["bf16"], a["rows"], a["N"], a["row_stride"], a["k"],
                            a["idx"], a["idx_stride"], None) == status


def test_fused_topk_workspace_bytes(lib):
    """The fused call's workspace holds per row a mask word per 32 keys of the
    filtered tiles, the threshold, the sampled tiles (one 128-key tile in four,
    4 bytes a key) and a value slot for every key of the other tiles, each part
    256-byte aligned."""
    def expect(B, S, N):
        tiles = -(-N // 128)
        st = -(-tiles // 4)
        ft = tiles - st
        rows = B * S
        a = lambda x: -(-x // 256) * 256
        off_thr = a(4 * ft * 4 * rows)
        off_s = a(off_thr + 4 * rows)
        off_c = a(off_s + 4 * rows * st * 128)
        return a(off_c + 4 * rows * ft * 128)
    for B, S, N in [(1, 1, 1), (1, 4, 127), (2, 40, 3000), (1, 8192, 65536), (3, 5, 513)]:
        assert binding.indexer_logits_topk_workspace_bytes(shp(B=B, S=S, N=N)) == expect(B, S, N)
    assert lib.indexer_logits_topk_workspace_bytes(None) == -1
    assert binding.indexer_logits_topk_workspace_bytes(shp(N=0)) == -1


@pytest.mark.parametrize("over,status", [
    (dict(idx=None), 1),
    (dict(workspace=None), 1),
    (dict(shape=None), 1),
    (dict(topk=0), 2),
    (dict(idx_stride=7), 2),                                 # < topk
    (dict(flags=2), 9),                                      # BF16 logits: no logits here
    (dict(workspace_bytes=1024), 10),                        # too small
    (dict(workspace=ctypes.c_void_p(0x1010)), 4),            # not 256-byte aligned
])
def test_fused_topk_host_validation(lib, over, status):
    shape = shp(flags=over.pop("flags", 0))
    a = dict(topk=8, idx=FAKE, idx_stride=8, workspace=ctypes.c_void_p(0x100000),
             workspace_bytes=1 << 40, shape=ctypes.byref(shape))
    a.update(over)
    assert lib.indexer_logits_topk(FAKE, None, FAKE, None, None, FAKE, FAKE, FAKE,
                                   ctypes.c_float(0.1), a["shape"], a["topk"], a["idx"],
                                   a["idx_stride"], a["workspace"], a["workspace_bytes"],
                                   None) == status


@pytest.mark.parametrize("over,status", [
    (dict(cu_q=None), 1),
    (dict(ke=None), 1),
    (dict(num_seqs=0), 2),
    (dict(total_q=0), 2),
    (dict(ks=ctypes.c_void_p(0x1002)), 4),
])
def test_thd_windows_host_validation(lib, over, status):
    a = dict(cu_q=FAKE, cu_k=FAKE, num_seqs=3, total_q=10, causal=1, ks=FAKE, ke=FAKE)
    a.update(over)
    assert lib.indexer_thd_windows(a["cu_q"], a["cu_k"], a["num_seqs"], a["total_q"],
                                   a["causal"], a["ks"], a["ke"], None) == status
