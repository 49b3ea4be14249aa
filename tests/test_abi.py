"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad host-side arguments before touching the GPU (no GPU needed)."""
import os
import re

import pytest

import tensor_program_compilers_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return pkg.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert names == sorted(pkg.EXPORTED), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (1, "ATTN_ERR_INVALID_ARG"), (2, "ATTN_ERR_ALIGNMENT"),
                       (3, "ATTN_ERR_UNSUPPORTED_DEVICE"), (4, "ATTN_ERR_CUDA"),
                       (5, "ATTN_ERR_TIMEOUT"), (6, "ATTN_ERR_BAD_SEQLENS")]:
        assert pkg.attn_status_string(code) == name
    assert pkg.attn_status_string(99) == "ATTN_UNKNOWN_STATUS"


def call(**kw):
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=2, Hq=8, Hkv=2, N=256,
                d=128, scale=0.088, causal=1, cu_seqlens=None, stream=0)
    args.update(kw)
    return pkg.attn_fwd(check=False, **args)


@pytest.mark.parametrize("kw", [
    dict(d=96), dict(d=32), dict(d=512), dict(Hq=6, Hkv=4), dict(Hkv=0), dict(Hq=0),
    dict(B=-1), dict(N=-5), dict(scale=0.0), dict(scale=-1.0), dict(scale=float("inf")),
    dict(scale=float("nan")), dict(q=None), dict(lse=None), dict(o=None),
    dict(N=1 << 30, B=4),          # more than 2^31 token rows
])
def test_invalid_arguments_rejected_without_gpu(lib, kw):
    assert call(**kw) == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(q=0x1008), dict(k=0x2004), dict(v=0x3002),
                                dict(o=0x4001), dict(lse=0x5002)])
def test_misaligned_pointers_rejected(lib, kw):
    assert call(**kw) == pkg.ATTN_ERR_ALIGNMENT


@pytest.mark.parametrize("kw", [dict(B=0), dict(N=0), dict(B=0, q=None, o=None)])
def test_empty_problem_is_a_no_op(lib, kw):
    assert call(**kw) == pkg.ATTN_OK


def test_selftest_rejects_bad_limit(lib):
    assert pkg.attn_selftest_timeout(0, stream=0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_selftest_timeout(2_000_000, stream=0) == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(scratch=None), dict(result=None), dict(hops=0),
                                dict(hops=2_000_000), dict(nbytes=1 << 20)])
def test_latency_probe_rejects_bad_arguments(lib, kw):
    args = dict(scratch=0x10000, nbytes=512 << 20, hops=100, result=0x20000, stream=0)
    args.update(kw)
    assert pkg.attn_probe_dram_latency(check=False, **args) == pkg.ATTN_ERR_INVALID_ARG


def test_latency_probe_rejects_misaligned_buffers(lib):
    assert pkg.attn_probe_dram_latency(0x10008, 512 << 20, 100, 0x20000, stream=0,
                                       check=False) == pkg.ATTN_ERR_ALIGNMENT
    assert pkg.attn_probe_dram_latency(0x10000, 512 << 20, 100, 0x20004, stream=0,
                                       check=False) == pkg.ATTN_ERR_ALIGNMENT


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(pkg, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        pkg.library()


def call_ex(window=None, softcap=0.0, alibi_slopes=None, **kw):
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=2, Hq=8, Hkv=2, N=256,
                d=128, scale=0.088, causal=1, cu_seqlens=None, stream=0)
    args.update(kw)
    return pkg.attn_fwd_ex(check=False, window=window, softcap=softcap,
                           alibi_slopes=alibi_slopes, **args)


@pytest.mark.parametrize("cap", [-1.0, float("inf"), float("nan")])
def test_variant_bad_softcap_rejected(lib, cap):
    assert call_ex(softcap=cap) == pkg.ATTN_ERR_INVALID_ARG


def test_variant_misaligned_slopes_rejected(lib):
    assert call_ex(alibi_slopes=0x6002) == pkg.ATTN_ERR_ALIGNMENT


@pytest.mark.parametrize("kw", [dict(B=0), dict(N=0)])
def test_variant_empty_problem_is_a_no_op(lib, kw):
    assert call_ex(window=(128, 0), softcap=30.0, alibi_slopes=0x6000, **kw) == pkg.ATTN_OK


def test_variant_struct_layout():
    """attn_variant is {int, int, float, const float *}: pointer at offset 16."""
    import ctypes
    assert ctypes.sizeof(pkg.AttnVariant) == 24
    assert pkg.AttnVariant.alibi_slopes.offset == 16


def call_dec(**kw):
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=2, Hq=8, Hkv=2, Nq=1,
                Nk=4096, d=128, scale=0.088, causal=0, seqlens_k=None, workspace=0x7000,
                workspace_bytes=1 << 20, stream=0)
    args.update(kw)
    return pkg.attn_fwd_decode(check=False, **args)


@pytest.mark.parametrize("kw", [
    dict(d=96), dict(Hq=6, Hkv=4), dict(Nq=33, Hq=8, Hkv=2),   # group x Nq > 128
    dict(Nq=5, Nk=4), dict(B=-1), dict(scale=0.0), dict(q=None), dict(lse=None),
    dict(Nk=1 << 30, B=4),
])
def test_decode_invalid_arguments_rejected_without_gpu(lib, kw):
    assert call_dec(**kw) == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(q=0x1008), dict(workspace=0x7004), dict(seqlens_k=0x6002)])
def test_decode_misaligned_pointers_rejected(lib, kw):
    assert call_dec(**kw) == pkg.ATTN_ERR_ALIGNMENT


@pytest.mark.parametrize("kw", [dict(B=0), dict(Nq=0)])
def test_decode_empty_problem_is_a_no_op(lib, kw):
    assert call_dec(**kw) == pkg.ATTN_OK


def call_paged(**kw):
    args = dict(q=0x1000, k_cache=0x2000, v_cache=0x3000, o=0x4000, lse=0x5000, B=2, Hq=8,
                Hkv=2, Nq=1, d=128, scale=0.088, causal=0, seqlens_k=0x6000,
                block_table=0x7000, max_blocks=64, page_size=64, num_pages=200,
                workspace=0x8000, workspace_bytes=1 << 20, stream=0)
    args.update(kw)
    return pkg.attn_fwd_decode_paged(check=False, **args)


@pytest.mark.parametrize("kw", [dict(page_size=8), dict(page_size=48), dict(page_size=96),
                                dict(page_size=200), dict(max_blocks=0), dict(num_pages=0),
                                dict(seqlens_k=None), dict(block_table=None), dict(d=80),
                                dict(Nq=40)])
def test_paged_invalid_arguments_rejected_without_gpu(lib, kw):
    assert call_paged(**kw) == pkg.ATTN_ERR_INVALID_ARG


def test_paged_misaligned_table_rejected(lib):
    assert call_paged(block_table=0x7002) == pkg.ATTN_ERR_ALIGNMENT


def test_paged_status_string(lib):
    assert pkg.attn_status_string(7) == "ATTN_ERR_BAD_PAGE_TABLE"


def call_bwd(**kw):
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, dout=0x5000, lse=0x6000, dq=0x7000,
                dk=0x8000, dv=0x9000, B=2, Hq=8, Hkv=2, N=256, d=128, scale=0.088, causal=1,
                cu_seqlens=None, workspace=0xA000, workspace_bytes=1 << 20, stream=0)
    args.update(kw)
    return pkg.attn_bwd(check=False, **args)


@pytest.mark.parametrize("kw", [dict(d=512), dict(d=96), dict(d=32), dict(Hq=6, Hkv=4), dict(scale=0.0),
                                dict(dq=None), dict(lse=None), dict(dout=None),
                                dict(workspace=None), dict(workspace_bytes=16),
                                dict(N=1 << 30, B=4)])
def test_bwd_invalid_arguments_rejected_without_gpu(lib, kw):
    assert call_bwd(**kw) == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(dq=0x7008), dict(dout=0x5004), dict(workspace=0xA004),
                                dict(lse=0x6002), dict(cu_seqlens=0xB002)])
def test_bwd_misaligned_pointers_rejected(lib, kw):
    assert call_bwd(**kw) == pkg.ATTN_ERR_ALIGNMENT


def test_bwd_workspace_size():
    # padded blocks: ceil(rows / 128) + B; two fp32 values per (head, padded row); B + 1 ints
    assert pkg.attn_bwd_workspace_bytes(2, 8, 300) == 2 * 8 * (5 + 2) * 128 * 4 + 3 * 4
    assert pkg.attn_bwd_workspace_bytes(3, 4, 1000, packed=True) == 2 * 4 * (8 + 3) * 128 * 4 + 16


def call_bwd_single(**kw):
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, dout=0x5000, lse=0x6000, dq=0x7000,
                dk=0x8000, dv=0x9000, B=2, Hq=8, Hkv=2, N=256, d=64, scale=0.125, causal=1,
                cu_seqlens=None, workspace=0xA000, workspace_bytes=1 << 24, stream=0)
    args.update(kw)
    return pkg.attn_bwd_single_pass(check=False, **args)


@pytest.mark.parametrize("kw", [dict(d=128), dict(d=256), dict(d=32), dict(Hq=6, Hkv=4),
                                dict(scale=0.0), dict(dq=None), dict(lse=None),
                                dict(workspace=None), dict(workspace_bytes=16),
                                # the two-kernel path's workspace (rows 512: 4 + 2
                                # padded blocks) is too small here
                                dict(workspace_bytes=2 * 8 * (4 + 2) * 128 * 4 + 3 * 4),
                                dict(N=1 << 30, B=4)])
def test_bwd_single_pass_invalid_arguments_rejected_without_gpu(lib, kw):
    assert call_bwd_single(**kw) == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(dq=0x7008), dict(dk=0x8004), dict(workspace=0xA008),
                                dict(lse=0x6002), dict(cu_seqlens=0xB002)])
def test_bwd_single_pass_misaligned_pointers_rejected(lib, kw):
    assert call_bwd_single(**kw) == pkg.ATTN_ERR_ALIGNMENT


@pytest.mark.parametrize("kw", [dict(B=0), dict(N=0)])
def test_bwd_single_pass_empty_problem_is_a_no_op(lib, kw):
    assert call_bwd_single(**kw) == pkg.ATTN_OK


def test_bwd_single_pass_workspace_size():
    # the fp32 dQ buffer (Hq x padded rows x 64) ahead of the two-kernel path's workspace
    for B, Hq, N, packed in ((2, 8, 300, False), (3, 4, 1000, True), (1, 1, 1, False)):
        rows = N if packed else B * N
        rows_pad = ((rows + 127) // 128 + B) * 128
        base = pkg.attn_bwd_workspace_bytes(B, Hq, N, packed=packed)
        assert pkg.attn_bwd_single_pass_workspace_bytes(B, Hq, N, packed=packed) == \
            Hq * rows_pad * 64 * 4 + base
    assert pkg.attn_bwd_single_pass_workspace_bytes(0, 8, 300) == 0
    assert pkg.attn_bwd_single_pass_workspace_bytes(2, 8, 0) == 0
