"""The C-ABI library: exports, struct layout and host-side validation (CPU only).

No kernel is launched here: every call below is rejected by the host checks
before any CUDA call is made, so these tests run without a GPU.
"""

import ctypes
import os
import re
import subprocess

import pytest

import compressed_mla_attention_gb300 as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsfm.h")


@pytest.fixture(scope="module")
def lib():
    from compressed_mla_attention_gb300 import build

    build.build()
    return Q.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsfm_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert "qsfm_forward" in names and "qsfm_metadata" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(Q.EXPORTS)
    # version 2 appended qsfm_params.kv_layout, version 3 the KV storage layouts and ori
    # picks, version 4 the lightning indexer's entry points
    assert lib.qsfm_abi_version() == 6


def test_exports_are_c_symbols(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", Q.LIB_PATH], capture_output=True, text=True).stdout
    for n in declared_functions():
        assert re.search(rf"\bT {n}$", out, flags=re.M), n


@pytest.mark.parametrize("cls,cname", [(Q.QsfmParams, "qsfm_params"), (Q.IndexerParams, "qsfm_indexer_params")])
def test_struct_layout_matches_c(tmp_path, cls, cname):
    src = tmp_path / "layout.c"
    fields = [f[0] for f in cls._fields_]
    body = "\n".join(f'  printf("{f} %zu\\n", offsetof({cname}, {f}));' for f in fields)
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "qsfm.h"\nint main(void){\n'
                   + body + f'\n  printf("sizeof %zu\\n", sizeof({cname}));\n  return 0;\n}}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(line.split() for line in out if line)
    for f in fields:
        assert int(got[f]) == getattr(cls, f).offset, f
    assert int(got["sizeof"]) == ctypes.sizeof(cls)


def test_params_init_defaults(lib):
    p = Q.QsfmParams()
    lib.qsfm_params_init(ctypes.byref(p))
    assert (p.n1, p.d, p.ori_block_size, p.cmp_ratio) == (64, 512, 128, 1)
    assert (p.ori_mask_mode, p.cmp_mask_mode, p.ori_win_left, p.ori_win_right) == (4, 3, 127, 0)
    assert abs(p.softmax_scale - 512 ** -0.5) < 1e-7


def _valid(lib):
    """A params struct that passes validation (fake non-null device pointers)."""
    p = Q.QsfmParams()
    lib.qsfm_params_init(ctypes.byref(p))
    p.batch, p.max_s1, p.num_ctas = 2, 1, 8
    p.ori_max_blocks, p.ori_num_blocks = 4, 8
    for f in ("q", "attn_out", "ori_kv", "ori_scale", "ori_block_table", "seqused_ori_kv", "metadata"):
        setattr(p, f, 0x1000)
    return p


def _status(lib, p, fn="qsfm_forward"):
    if fn == "qsfm_forward":
        return lib.qsfm_forward(ctypes.byref(p), None, 0, None)
    if fn == "qsfm_metadata":
        return lib.qsfm_metadata(ctypes.byref(p), None, None)
    n = ctypes.c_size_t(0)
    return lib.qsfm_forward_workspace_size(ctypes.byref(p), ctypes.byref(n))


INVALID = [
    ("d != 512", dict(d=256), 1),
    ("n1 = 96 is not built (the pages allow 64 and 128)", dict(n1=96), 2),
    ("n1 = 0", dict(n1=0), 1),
    ("block size 64 not built", dict(ori_block_size=64), 2),
    ("block size 2048 invalid", dict(ori_block_size=2048), 1),
    ("cmp_ratio 0", dict(cmp_ratio=0), 1),
    ("cmp_ratio 129", dict(cmp_ratio=129), 1),
    ("cmp_ratio != 1 without cmp_kv", dict(cmp_ratio=4), 1),
    ("ori mask mode 2", dict(ori_mask_mode=2), 1),
    ("cmp mask mode 4", dict(cmp_mask_mode=4), 1),
    ("window < -1", dict(ori_win_left=-2), 1),
    ("window >= 0 with mode 3", dict(ori_mask_mode=3, ori_win_left=5, ori_win_right=-1), 1),
    ("window >= 0 with mode 0", dict(ori_mask_mode=0, ori_win_left=-1, ori_win_right=0), 1),
    ("TND without cu_seqlens_q", dict(layout_q=1, total_t=4), 1),
    ("bad layout", dict(layout_q=7), 1),
    ("no seqused_ori_kv", dict(seqused_ori_kv=None), 1),
    ("no ori block table", dict(ori_block_table=None), 1),
    ("no ori scale", dict(ori_scale=None), 1),
    ("indices without cmp_kv", dict(cmp_sparse_indices=0x1000, k2=512), 1),
    ("no q", dict(q=None), 1),
    ("no output", dict(attn_out=None), 1),
    ("lse requested without buffer", dict(return_lse=1), 1),
    ("no metadata", dict(metadata=None), 1),
    ("too many CTAs", dict(num_ctas=100000), 1),
    ("nan scale", dict(softmax_scale=float("nan")), 1),
    ("q not 16-byte aligned", dict(q=0x1008), 1),
    ("ori_kv not 16-byte aligned", dict(ori_kv=0x1004), 1),
    ("attn_out not 16-byte aligned", dict(attn_out=0x1002), 1),
    ("ori_scale not 4-byte aligned", dict(ori_scale=0x1002), 1),
    ("block table not 4-byte aligned", dict(ori_block_table=0x1001), 1),
    ("metadata not 4-byte aligned", dict(metadata=0x1003), 1),
]


@pytest.mark.parametrize("why,change,code", INVALID, ids=[c[0] for c in INVALID])
def test_forward_rejects_invalid_arguments(lib, why, change, code):
    p = _valid(lib)
    for k, v in change.items():
        setattr(p, k, v)
    assert _status(lib, p) == code


def test_cmp_side_requirements(lib):
    p = _valid(lib)
    p.cmp_kv, p.cmp_ratio = 0x1000, 4
    assert _status(lib, p) == 1  # no cmp scale / table
    p.cmp_scale, p.cmp_block_table, p.cmp_max_blocks, p.cmp_num_blocks = 0x1000, 0x1000, 2, 4
    p.cmp_sparse_indices, p.k2 = 0x1000, 0
    assert _status(lib, p) == 1  # CSA needs K2 >= 1
    p.cmp_block_size = 256
    assert _status(lib, p, "size") == 2


def test_null_params_and_outputs(lib):
    assert lib.qsfm_forward(None, None, 0, None) == 1
    assert lib.qsfm_metadata(ctypes.byref(_valid(lib)), None, None) == 1  # no metadata_out
    assert lib.qsfm_forward_workspace_size(ctypes.byref(_valid(lib)), None) == 1
    assert lib.qsfm_get_device_status(None) == 1


def test_workspace_size_depends_on_split(lib):
    p = _valid(lib)
    n = ctypes.c_size_t(123)
    p.batch, p.max_s1, p.num_ctas = 2, 1, 8  # 2 tokens < 8 CTAs: tokens may be split
    assert lib.qsfm_forward_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value >= 2 * 8 * 64 * 512 * 4
    p.batch, p.max_s1 = 64, 1  # 64 tokens >= 8 CTAs: no split, no workspace
    assert lib.qsfm_forward_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 0


def test_kv_layout_checks(lib):
    p = _valid(lib)
    p.kv_layout = 1  # packed rows carry their scales: a separate scale tensor is an error
    assert _status(lib, p) == 1
    p.ori_scale = None
    assert _status(lib, p) == 4  # valid; stops at the missing workspace
    p.kv_layout = 2  # bf16 rows: no scales either
    assert _status(lib, p) == 4
    p.ori_scale = 0x2000
    assert _status(lib, p) == 1
    p.ori_scale = None
    p.kv_layout = 7
    assert _status(lib, p) == 1


def _non_paged(lib, layout_kv):
    """Valid params with non-paged ori KV (BSND with BSND q, TND with TND q)."""
    p = _valid(lib)
    p.ori_block_table = None
    p.layout_kv = Q.LAYOUT_KV[layout_kv]
    p.ori_kv_len = 100
    if layout_kv == "TND":
        p.layout_q, p.total_t, p.cu_seqlens_q = 1, 2, 0x1000
        p.seqused_ori_kv, p.cu_seqlens_ori_kv = None, 0x1000
    return p


NON_PAGED_INVALID = [
    ("BSND KV with TND q", "BSND", dict(layout_q=1, total_t=2, cu_seqlens_q=0x1000)),
    ("TND KV with BSND q", "TND", dict(layout_q=0, max_s1=1)),
    ("BSND KV with a block table", "BSND", dict(ori_block_table=0x1000)),
    ("BSND KV with no length", "BSND", dict(ori_kv_len=0)),
    ("BSND KV with cu_seqlens_ori_kv", "BSND", dict(cu_seqlens_ori_kv=0x1000)),
    ("TND KV without cu_seqlens_ori_kv", "TND", dict(cu_seqlens_ori_kv=None)),
    ("TND KV with seqused_ori_kv", "TND", dict(seqused_ori_kv=0x1000)),
    ("TND KV cmp without cu_seqlens_cmp_kv", "TND", dict(cmp_kv=0x1000, cmp_ratio=4, cmp_scale=0x1000,
                                                        cmp_kv_len=10)),
    ("TND KV cmp without length", "TND", dict(cmp_kv=0x1000, cmp_ratio=4, cmp_scale=0x1000,
                                              cu_seqlens_cmp_kv=0x1000)),
    ("cu_seqlens_cmp_kv without cmp_kv", "TND", dict(cu_seqlens_cmp_kv=0x1000)),
    ("layout_kv 3", "BSND", dict(layout_kv=3)),
    ("ori picks without K1", "BSND", dict(ori_sparse_indices=0x1000)),
    ("K1 without ori picks", "BSND", dict(k1=8)),
    ("ori_topk_length without ori picks", "BSND", dict(ori_topk_length=0x1000)),
    ("ori picks not 4-byte aligned", "BSND", dict(ori_sparse_indices=0x1002, k1=8)),
    ("cu_seqlens_ori_kv not 4-byte aligned", "TND", dict(cu_seqlens_ori_kv=0x1001)),
]


@pytest.mark.parametrize("why,layout_kv,change", NON_PAGED_INVALID, ids=[c[0] for c in NON_PAGED_INVALID])
def test_non_paged_kv_and_ori_picks_rules(lib, why, layout_kv, change):
    p = _non_paged(lib, layout_kv)
    assert _status(lib, p, "size") == 0, "the base case must be valid"
    for k, v in change.items():
        setattr(p, k, v)
    assert _status(lib, p, "size") == 1


def test_non_paged_kv_and_ori_picks_valid_cases(lib):
    p = _non_paged(lib, "BSND")
    p.seqused_ori_kv = None  # optional for BSND KV
    p.ori_sparse_indices, p.k1, p.ori_topk_length = 0x1000, 512, 0x2000
    p.cmp_kv, p.cmp_ratio, p.cmp_scale, p.cmp_kv_len = 0x1000, 4, 0x1000, 25
    assert _status(lib, p, "size") == 0
    p = _non_paged(lib, "TND")
    p.cmp_kv, p.cmp_ratio, p.cmp_scale, p.cmp_kv_len, p.cu_seqlens_cmp_kv = 0x1000, 4, 0x1000, 25, 0x1000
    assert _status(lib, p, "size") == 0
    p = _valid(lib)  # paged KV with ori picks
    p.ori_sparse_indices, p.k1 = 0x1000, 64
    assert _status(lib, p, "size") == 0
    p.k1 = 1 << 17
    assert _status(lib, p, "size") == 2  # K1 past the index limit


def test_bsnd_kv_row_limit_is_refused(lib):
    p = _non_paged(lib, "BSND")
    p.batch, p.ori_kv_len = 1 << 10, 1 << 21  # 2^31 rows
    assert _status(lib, p, "size") == 2


def test_debug_gather_argument_rules(lib):
    """Row bytes are exported in every row format; separate scales exist for
    fp8 rows only. Every case below is refused on the host (no launch)."""
    p = _valid(lib)
    # fp8 rows: rows and scales go together
    assert lib.qsfm_debug_gather(ctypes.byref(p), 0x1000, 1, 1, 0x1000, None, 0x1000, 0x1000, None) == 1
    assert lib.qsfm_debug_gather(ctypes.byref(p), 0x1000, 1, 1, None, 0x1000, 0x1000, 0x1000, None) == 1
    # row bytes must be 16-byte aligned
    assert lib.qsfm_debug_gather(ctypes.byref(p), 0x1000, 1, 1, 0x1008, 0x1000, 0x1000, 0x1000, None) == 1
    for layout in (1, 2):
        p.kv_layout, p.ori_scale = layout, None
        # packed and bf16 rows have no separate scales to export
        assert lib.qsfm_debug_gather(ctypes.byref(p), 0x1000, 1, 1, 0x1000, 0x1000, 0x1000, 0x1000, None) == 1
        # row ids (with or without row bytes) need the id buffer
        assert lib.qsfm_debug_gather(ctypes.byref(p), 0x1000, 1, 1, None, None, None, 0x1000, None) == 1
        assert lib.qsfm_debug_gather(ctypes.byref(p), 0x1000, 1, 1, 0x1000, None, None, 0x1000, None) == 1


def test_noalloc_scratch_size_matches_header():
    """The binding reads the scratch size from the C header, not a copy."""
    import re

    import compressed_mla_attention_gb300 as Q

    text = open(os.path.join(ROOT, "include", "qsfm.h")).read()
    m = re.search(r"#define QSFM_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m is not None
    assert Q.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


@pytest.mark.parametrize("why,change", [
    ("2^24 + 1 units", dict(batch=(1 << 24) + 1, max_s1=1)),
    ("2^23 + 1 tokens of 128 heads", dict(batch=(1 << 23) + 1, max_s1=1, n1=128)),
    ("k2 above 65536", dict(k2=(1 << 16) + 1)),
    ("2^31 rows in the ori pool", dict(ori_num_blocks=1 << 24)),
])
def test_index_limits_are_refused(lib, why, change):
    # qsfm_forward_workspace_size validates like qsfm_forward and never launches
    p = _valid(lib)
    for k, v in change.items():
        setattr(p, k, v)
    assert _status(lib, p, fn="workspace") == 2, why  # QSFM_ERR_UNSUPPORTED


def test_index_limits_allow_the_largest_shapes(lib):
    p = _valid(lib)
    p.batch, p.max_s1, p.k2, p.ori_num_blocks = 1 << 23, 2, 1 << 16, (1 << 24) - 1
    assert _status(lib, p, fn="workspace") == 0  # validation only, nothing launched


def test_n1_128_passes_validation(lib):
    p = _valid(lib)
    p.n1 = 128
    assert _status(lib, p) == 4  # valid; stops at the missing workspace (4 units < 8 CTAs split)


def test_word_aligned_pointers_pass_validation(lib):
    # 4-byte alignment is enough for scales, tables and lengths: validation
    # passes and the call stops at the missing workspace instead
    p = _valid(lib)
    p.ori_scale, p.ori_block_table, p.seqused_ori_kv, p.metadata = 0x1004, 0x1008, 0x100C, 0x1004
    assert _status(lib, p) == 4
    plan = ctypes.c_void_p(0x1002)
    assert lib.qsfm_metadata(ctypes.byref(_valid(lib)), plan, None) == 1


def test_forward_needs_workspace_when_splitting(lib):
    p = _valid(lib)
    assert lib.qsfm_forward(ctypes.byref(p), None, 0, None) == 4


def test_debug_bounded_wait_rejects_bad_arguments(lib):
    assert lib.qsfm_debug_bounded_wait(1000, None, None) == 1          # no output
    assert lib.qsfm_debug_bounded_wait(0, 0x1000, None) == 1           # no limit
    assert lib.qsfm_debug_bounded_wait(2_000_000_000, 0x1000, None) == 1  # over one second
    assert lib.qsfm_debug_bounded_wait(1000, 0x1004, None) == 1        # misaligned output


def test_status_strings(lib):
    for code in range(7):
        assert Q.status_string(code)
    assert "invalid" in Q.status_string(1)


def _indexer_valid(lib):
    p = Q.IndexerParams()
    lib.qsfm_indexer_params_init(ctypes.byref(p))
    p.batch, p.max_s1, p.topk, p.max_blocks, p.num_blocks = 2, 1, 512, 4, 8
    for f in ("query", "query_scale", "weights", "key", "key_scale", "block_table", "seqused_k", "sparse_indices"):
        setattr(p, f, 0x1000)
    return p


def test_indexer_params_init_defaults(lib):
    p = Q.IndexerParams()
    lib.qsfm_indexer_params_init(ctypes.byref(p))
    assert (p.heads, p.dim, p.topk, p.block_size, p.mask_mode, p.cmp_ratio, p.layout_q) == (64, 128, 2048, 128, 0, 1, 0)


INDEXER_INVALID = [
    ("heads 0", dict(heads=0), 1), ("heads 65", dict(heads=65), 1), ("topk 0", dict(topk=0), 1),
    ("topk 8193", dict(topk=8193), 1), ("dim 64 not built", dict(dim=64), 2),
    ("block 64 not built", dict(block_size=64), 2), ("mask mode 4", dict(mask_mode=4), 1),
    ("cmp_ratio 0", dict(cmp_ratio=0), 1), ("cmp_ratio 129", dict(cmp_ratio=129), 1),
    ("BSND with cu_seqlens_q", dict(cu_seqlens_q=0x1000), 1),
    ("TND without cu_seqlens_q", dict(layout_q=1, total_t=4), 1),
    ("no query", dict(query=None), 1), ("no key scale", dict(key_scale=None), 1),
    ("no block table", dict(block_table=None), 1), ("no seqused_k", dict(seqused_k=None), 1),
    ("no output", dict(sparse_indices=None), 1), ("values without buffer", dict(return_value=1), 1),
    ("key not 16-byte aligned", dict(key=0x1008), 1), ("key scale not 16-byte aligned", dict(key_scale=0x1004), 1),
    ("weights not 4-byte aligned", dict(weights=0x1002), 1), ("no blocks", dict(num_blocks=0), 1),
    ("key layout 3", dict(layout_k=3), 1), ("paged keys with cu_seqlens_k", dict(cu_seqlens_k=0x1000), 1),
    ("BSND keys with a block table", dict(layout_k=1, max_sk=300), 1),
    ("TND keys without cu_seqlens_k", dict(layout_k=2, total_k=900, block_table=None, seqused_k=None), 1),
    ("TND keys with seqused_k", dict(layout_k=2, total_k=900, block_table=None, cu_seqlens_k=0x1000), 1),
    ("offsets not 4-byte aligned", dict(output_idx_offset=0x1002), 1),
]


@pytest.mark.parametrize("why,change,code", INDEXER_INVALID, ids=[c[0] for c in INDEXER_INVALID])
def test_indexer_rejects_invalid_arguments(lib, why, change, code):
    p = _indexer_valid(lib)
    for k, v in change.items():
        setattr(p, k, v)
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), 0x1000, 1 << 30, None) == code


def _indexer_ws(lib, p):
    n = ctypes.c_size_t(0)
    assert lib.qsfm_lightning_indexer_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    return n.value


def test_indexer_workspace_size(lib):
    """One fp32 row of min(32768, max_blocks * 128) scores per query row."""
    p = _indexer_valid(lib)
    assert _indexer_ws(lib, p) == 2 * 4 * 128 * 4
    p.max_blocks, p.batch, p.max_s1 = 1000, 3, 2
    assert _indexer_ws(lib, p) == 6 * 32768 * 4
    p.layout_q, p.total_t, p.cu_seqlens_q = 1, 5, 0x1000
    assert _indexer_ws(lib, p) == 5 * 32768 * 4
    p.heads = 0
    assert lib.qsfm_lightning_indexer_workspace_size(ctypes.byref(p), ctypes.byref(ctypes.c_size_t())) == 1
    assert lib.qsfm_lightning_indexer_workspace_size(ctypes.byref(p), None) == 1


def test_indexer_rejects_missing_or_small_workspace(lib):
    p = _indexer_valid(lib)
    need = _indexer_ws(lib, p)
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), None, need, None) == 4
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), 0x1000, need - 1, None) == 4
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), 0x1008, need, None) == 4


def test_indexer_rejects_too_many_query_rows(lib):
    p = _indexer_valid(lib)
    p.batch, p.max_s1 = 1 << 11, 1 << 10
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), 0x1000, 1 << 40, None) == 2


def test_indexer_tnd_takes_seqused_q(lib):
    """TND with seqused_q is TND padding (QuantLightningIndexerV2, 约束说明):
    accepted; only the workspace check is left to fail here."""
    p = _indexer_valid(lib)
    p.layout_q, p.total_t, p.cu_seqlens_q, p.seqused_q = 1, 4, 0x1000, 0x1000
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), None, 0, None) == 4


def test_indexer_empty_call_is_ok(lib):
    p = _indexer_valid(lib)
    p.batch = 0
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), None, 0, None) == 0
    assert lib.qsfm_lightning_indexer(None, None, 0, None) == 1


def test_last_cuda_error_starts_clear(lib):
    name = ctypes.c_char_p()
    assert lib.qsfm_last_cuda_error(ctypes.byref(name)) == 0
    assert name.value == b"cudaSuccess"
    assert lib.qsfm_last_cuda_error(None) == 0


@pytest.mark.parametrize("change", [dict(layout_k=1, max_sk=300, block_table=None),
                                    dict(layout_k=1, max_sk=300, block_table=None, seqused_k=None),
                                    dict(layout_k=2, total_k=900, block_table=None, seqused_k=None,
                                         cu_seqlens_k=0x1000, output_idx_offset=0x1000)],
                         ids=["BSND keys", "BSND keys without seqused_k", "TND keys with offsets"])
def test_indexer_non_paged_keys_are_accepted(lib, change):
    """BSND and TND key layouts (parameter table: layout_k) pass validation:
    only the missing workspace is refused."""
    p = _indexer_valid(lib)
    for k, v in change.items():
        setattr(p, k, v)
    assert lib.qsfm_lightning_indexer(ctypes.byref(p), None, 0, None) == 4
    n = ctypes.c_size_t(0)
    assert lib.qsfm_lightning_indexer_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 2 * (384 if change["layout_k"] == 1 else 1024) * 4
