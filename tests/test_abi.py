"""CPU-side checks of the C ABI: the library loads, exports every entry point
that include/sa.h declares, and rejects bad arguments on the host before any
CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                                 src, flags=re.M)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("csa_compress", "csa_index_topk", "csa_attend", "hca_compress_attend", "attn_merge"):
        assert n in names, names


def test_library_exports_every_declared_symbol():
    import sparse_attention_27_b300 as m
    lib = ctypes.CDLL(m.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(m.EXPORTS)


def test_status_strings_and_host_validation():
    import sparse_attention_27_b300 as m
    assert m.status_string(0) == "ok"
    assert "range" in m.status_string(m.SA_ERR_BOUNDS)
    # bad dtype / null pointers / R < W: rejected before any CUDA call
    with pytest.raises(m.SaError) as e:
        m.csa_compress(9, 9, 1, 128, 64, 4, None, None, None, None, 128, None, None, 1, None,
                       None, None, None, 10, stream=0)
    assert e.value.status == m.SA_ERR_INVALID_ARG
    with pytest.raises(m.SaError) as e:
        m.csa_attend(m.SA_BF16, 1, 1, 64, 128, 4, 8, 16, 0.1, None, None, None, None, 4, None,
                     None, None, 8, None, None, stream=0)
    assert e.value.status == m.SA_ERR_INVALID_ARG
    assert m.library().attn_merge(0, None, None, 1, 1, None, 0, None, None, None) == \
        m.SA_ERR_INVALID_ARG


def test_workspace_queries_are_host_only():
    import sparse_attention_27_b300 as m
    assert m.csa_index_topk_workspace_bytes(32, 1, 32768, 2048) == 32 * 32768 * 4
    assert m.csa_index_topk_workspace_bytes(0, 1, 10, 1) == 0


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="stand-in pointers: run only where no kernel can be launched")
def test_mxfp4_index_host_validation():
    """The MXFP4 scoring path's limits are checked on the host, before any
    launch: N_cap a multiple of 8 (every bulk copy of scales a multiple of 16
    bytes), both scale arrays given, 64 heads of width 64, 16-byte aligned
    operands.  Stand-in pointer values (16-byte aligned integers) are never
    dereferenced on these paths."""
    import sparse_attention_27_b300 as m
    P = 1 << 20                       # aligned stand-in address

    def call(N_cap=4096, HI=64, dI=64, q=P, qs=P, ik=P, iks=P):
        return m.library().csa_index_topk(m.SA_MXFP4, 2, 1, HI, dI, 4, 0, q, qs, P, ik, iks,
                                          N_cap, P, None, P, None, None, 0, None, None)
    assert call(N_cap=4100) == m.SA_ERR_UNSUPPORTED         # not a multiple of 8
    assert call(qs=None) == m.SA_ERR_UNSUPPORTED            # query scales missing
    assert call(iks=None) == m.SA_ERR_UNSUPPORTED           # key scales missing
    assert call(HI=32) == m.SA_ERR_UNSUPPORTED
    assert call(dI=128) == m.SA_ERR_UNSUPPORTED
    assert call(q=P + 8) == m.SA_ERR_INVALID_ARG            # codes not 16-byte aligned
    assert call(ik=None) == m.SA_ERR_INVALID_ARG


def _sms_148():
    return (not torch.cuda.is_available() or
            torch.cuda.get_device_properties(0).multi_processor_count == 148)


@pytest.mark.skipif(not _sms_148(), reason="split sizes below are worked out for 148 SMs")
def test_attention_workspace_queries_follow_the_split_rule():
    """Workspace sizes of the attention calls, worked out by hand from the split
    rule: key lists of 64-key tiles; the tensor-core kernel aims at 2 (row,
    split) items per SM, with no cap on a split's length; split s has
    ceil(tiles / ns) tiles; partials are rows*nsplit*H*d f32 for O plus
    rows*nsplit*H f32 for LSE, each rounded up to 256 B, then 256 B for the
    tensor-core kernel's item counter.  148 SMs (the count the library
    assumes without a device)."""
    import sparse_attention_27_b300 as m

    def ws(rows, nsplit, H=64, d=128):
        r256 = lambda x: (x + 255) // 256 * 256
        parts = r256(4 * rows * nsplit * H * d) + r256(4 * rows * nsplit * H) if nsplit > 1 else 0
        return parts + 256
    # 128K decode CSA: 32 rows, 2048/64 + 128/64 = 34 tiles; want ceil(296/32) = 10
    # splits -> 4 tiles each -> 9 splits
    assert m.csa_attend_workspace_bytes(m.SA_BF16, 32, 1, 64, 128, 2048, 128) == ws(32, 9)
    # 128K decode HCA: 1024/64 + 2 = 18 tiles; 10 wanted -> 2 tiles each -> 9 splits
    assert m.hca_compress_attend_workspace_bytes(m.SA_BF16, 32, 1, 64, 128, 1024, 128) == ws(32, 9)
    # 1M decode CSA: 4 rows want 74 splits, 34 tiles -> one tile each -> 34 splits
    assert m.csa_attend_workspace_bytes(m.SA_BF16, 4, 1, 64, 128, 2048, 128) == ws(4, 34)
    # 1M decode HCA: 8192/64 + 2 = 130 tiles; 74 wanted -> 2 tiles each -> 65 splits
    assert m.hca_compress_attend_workspace_bytes(m.SA_BF16, 4, 1, 64, 128, 8192, 128) == ws(4, 65)
    # 64K prefill CSA: 65536 rows fill the SMs, one split of 34 tiles, no partials
    assert m.csa_attend_workspace_bytes(m.SA_BF16, 1, 65536, 64, 128, 2048, 128) == ws(65536, 1)
    # fp32 (CUDA-core kernel, one item per CTA): 256 rows fill the SMs, no split
    assert m.csa_attend_workspace_bytes(m.SA_F32, 1, 256, 16, 128, 64, 128) == ws(256, 1)


def test_noalloc_limit_matches_the_header():
    """The Python binding's copy of the no-allocation call's size limit is the
    value include/sa.h gives the library's device array."""
    import sparse_attention_27_b300 as m
    src = open(os.path.join(ROOT, "include", "sa.h")).read()
    got = re.search(r"#define\s+SA_NOALLOC_MAX_SCORES\s+(\d+)", src)
    assert got is not None
    assert int(got.group(1)) == m.NOALLOC_MAX_SCORES


def test_decode_step_workspace_follows_its_layout():
    """sa_decode_step's workspace, worked by hand from its layout for the 128K
    decode (B=32, N_cap=32768, k=2048, W=128, N2_cap=1024; every part rounded
    up to 256 bytes):
      counters 32 + 7 per row (rounded up to 64 ints), then per row a 8192-bin
      histogram and 16 ints of top-k info:  4 * (256 + 32 * 8208)   = 1051648
      score keys, rows of 32768:            4 * 32 * 32768          = 4194304
      CSA shares: 34 key tiles -> 4 shares  4 * 32 * 4 * 64 * 128   = 4194304
        and their LSEs                      4 * 32 * 4 * 64         =   32768
      HCA shares: 18 key tiles -> 2 shares  4 * 32 * 2 * 64 * 128   = 2097152
        and their LSEs                      4 * 32 * 2 * 64         =   16384
      top-k candidate lists, 4 x 4096/row   4 * 32 * 4 * 4096       = 2097152
    Rows longer than 32768 entries (the 1M decode) are not taken: 0."""
    m = pytest.importorskip("sparse_attention_27_b300")
    assert m.sa_decode_step_workspace_bytes(32, 64, 32768, 2048, 128, 1024) == (
        1051648 + 4194304 + 4194304 + 32768 + 2097152 + 16384 + 2097152)
    assert m.sa_decode_step_workspace_bytes(4, 64, 262144, 2048, 128, 8192) == 0
    assert m.sa_decode_step_workspace_bytes(0, 64, 100, 64, 16, 4) == 0
