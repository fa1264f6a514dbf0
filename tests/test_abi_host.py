"""Host-side checks of the C ABI (no GPU needed: nothing here launches work).

The library must load on a machine without a GPU, export every function the
header declares, and reject bad arguments on the host before any CUDA call.
"""
import ctypes
import os
import re

import pytest

import paged_kv_attention_decode_gb300 as pa
from paged_kv_attention_decode_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_binding.library_path()):
        from paged_kv_attention_decode_gb300 import build_lib
        build_lib.build()
    return _binding.load_library()


def header_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_path(lib):
    names = header_functions()
    for want in ("pa_slot_mapping", "pa_paged_kv_write", "pa_paged_attention_decode",
                 "pa_paged_attention_prefill", "pa_decode_workspace_bytes", "pa_get_device_error",
                 "pa_copy_blocks", "pa_bm_create", "pa_bm_allocate_slots", "pa_bm_build_step"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_binding.library_path())
    missing = [n for n in header_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert lib.pa_version() >= 100
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(3) == b"PA_ERR_WORKSPACE_TOO_SMALL"
    assert lib.pa_status_string(99) == b"PA_ERR_UNKNOWN"


def _align(x):
    return (x + 255) // 256 * 256


def _partials(rows, heads, parts, dim=128):
    n = rows * heads * parts
    return 2 * _align(n * 4) + _align(n * dim * 4)


def test_automatic_partition(lib):
    # 512 tokens, doubled while a max_seq_len sequence would have more than 64 partitions
    assert pa.decode_partition(0) == 512
    assert pa.decode_partition(4096) == 512
    assert pa.decode_partition(32768) == 512          # exactly 64 partitions
    assert pa.decode_partition(32769) == 1024
    assert pa.decode_partition(131072) == 2048
    assert pa.decode_partition(131073) == 4096
    assert pa.decode_partition(10 ** 8) == 8192       # capped
    assert pa.decode_partition(131072, 256) == 256    # an explicit length is kept
    for bad in ((-1, 0), (4096, 100), (4096, -16)):
        with pytest.raises(pa.PagedAttnError):
            pa.decode_partition(*bad)


def test_workspace_sizes(lib):
    # [header 256 B][work list: B x partitions int32]
    # + when partitions > 1: [row_base: B int32][rows: R int32][partials of R rows]
    assert pa.decode_workspace_bytes(64, 32, 128, 512, 512) == 256 + _align(64 * 4)
    assert pa.decode_workspace_bytes(64, 32, 128, 4096, 512) == (256 + _align(64 * 8 * 4) + _align(64 * 4)
                                                                 + _align(64 * 4) + _partials(64, 32, 8))
    # 131072 tokens: the automatic partition is 2048 tokens (64 partitions)
    assert pa.decode_workspace_bytes(8, 64, 128, 131072, 0) == (256 + _align(8 * 64 * 4) + 2 * _align(8 * 4)
                                                                + _partials(8, 64, 64))
    assert pa.decode_workspace_bytes(8, 64, 128, 131072, 512) == (256 + _align(8 * 256 * 4) + 2 * _align(8 * 4)
                                                                  + _partials(8, 64, 256))
    # prefill: [plan: offsets (B + 1) + cost-sorted pair list (T / 4 + B) int32]
    # + the decode part, partials rows = min(num_tokens, 8 * num_seqs) (decode and verify chunks)
    def _plan(B, T):
        # offsets, then two pair lists (the cost order, each pair's sequence)
        return _align((B + 1 + 2 * (T // 4 + B)) * 4)
    assert pa.prefill_workspace_bytes(8, 8, 64, 128, 131072) == (_plan(8, 8)
                                                                 + pa.decode_workspace_bytes(8, 64, 128, 131072, 0))
    assert pa.prefill_workspace_bytes(8, 6000, 64, 128, 131072) == (_plan(8, 6000) + 256 + _align(8 * 64 * 4)
                                                                    + _align(8 * 4) + _align(64 * 4)
                                                                    + _partials(64, 64, 64))
    assert pa.prefill_workspace_bytes(4, 12, 32, 128, 1024) == (_plan(4, 12) + 256 + _align(4 * 2 * 4)
                                                                + _align(4 * 4) + _align(12 * 4)
                                                                + _partials(12, 32, 2))
    assert pa.prefill_workspace_bytes(2052, 8192, 32, 128, 300) == _plan(2052, 8192) + 256 + _align(2052 * 4)
    assert pa.prefill_workspace_bytes(0, 0, 32, 128, 300) == 0
    assert pa.prefill_workspace_bytes(4, -1, 32, 128, 300) == 0
    assert pa.decode_workspace_bytes(0, 32, 128, 300, 0) == 0


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced on rejected calls


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, maxb=4, sl=FAKE, B=2, maxlen=64, nb=8,
             scale=0.1, hq=4, hkv=2, d=128, bs=16, part=0, ws=None, wsb=0, dt=0)
    a.update(kw)
    return lib.pa_paged_attention_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["maxb"], a["sl"],
                                         a["B"], a["maxlen"], a["nb"], a["scale"], a["hq"], a["hkv"],
                                         a["d"], a["bs"], a["part"], a["ws"], a["wsb"], a["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(dt=7), 2), (dict(d=96), 2), (dict(bs=32), 2), (dict(hq=5, hkv=2), 1),
    (dict(hq=65, hkv=1), 2), (dict(hq=64, hkv=1), 3), (dict(part=17), 1), (dict(part=-16), 1), (dict(q=None), 1),
    (dict(out=FAKE + 2), 1), (dict(B=-1), 1), (dict(nb=0), 1), (dict(scale=float("nan")), 1),
    (dict(maxlen=4096, part=512), 3), (dict(maxlen=4096, ws=FAKE, wsb=10), 3), (dict(maxlen=16), 3),
    (dict(maxlen=1 << 24, part=16), 1),
    (dict(B=0), 0),
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_write_and_slot_mapping_reject_bad_arguments(lib):
    w = lib.pa_paged_kv_write
    assert w(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 96, 16, 0, None) == 2
    assert w(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 128, 8, 0, None) == 2
    assert w(FAKE, FAKE, FAKE, FAKE, None, 4, 8, 2, 128, 16, 0, None) == 1
    assert w(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 2, 128, 16, 0, None) == 0
    s = lib.pa_slot_mapping
    assert s(FAKE, FAKE, 4, FAKE, None, 3, 5, 8, 16, None) == 1     # decode form needs T == B
    assert s(FAKE, FAKE, 4, FAKE, None, 3, 3, 8, 32, None) == 2
    assert s(FAKE, FAKE, 4, FAKE, None, 0, 0, 8, 16, None) == 0


def test_prefill_rejects_bad_arguments(lib):
    p = lib.pa_paged_attention_prefill
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 10, 8, 64, 8, 0.1, 8, 2, 128, 16, None, 0, 1, None]
    bad = list(args)
    bad[7] = None        # cu_q_lens
    assert p(*bad) == 1
    bad = list(args)
    bad[14], bad[15] = 9, 3   # group 3 is fine, 9 % 3 == 0, but check head_dim
    bad[16] = 80
    assert p(*bad) == 2


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(_binding.PagedAttnError):
        _binding.load_library()


def test_copy_blocks_rejects_bad_arguments_on_the_host(lib):
    f = lib.pa_copy_blocks
    assert f(FAKE, FAKE, FAKE, -1, 8, 8, 128, 2, None) == 1         # negative pair count
    assert f(FAKE, FAKE, FAKE, 1, 0, 8, 128, 2, None) == 1          # empty pool
    assert f(FAKE, FAKE, FAKE, 1, 8, 8, 128, 4, None) == 2          # 4-byte elements
    assert f(FAKE, FAKE, None, 1, 8, 8, 128, 2, None) == 1          # no pair list
    assert f(FAKE + 8, FAKE, FAKE, 1, 8, 8, 128, 2, None) == 1      # misaligned pool
    assert f(None, None, None, 0, 8, 8, 128, 2, None) == 0          # nothing to copy


def test_fp8_entry_points_reject_bad_arguments_on_the_host(lib):
    w = lib.pa_paged_kv_write_fp8
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 128, 16, 0, 1.0, 1.0, None]

    def write(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return w(*a)

    assert write(a8=64) == 2                 # head_dim must be 128
    assert write(a9=32) == 2                 # block size
    assert write(a10=5) == 2                 # source dtype
    assert write(a11=0.0) == 1 and write(a12=-1.0) == 1 and write(a11=float("inf")) == 1
    assert write(a4=None) == 1               # slot mapping
    assert write(a5=0) == 0                  # nothing to write
    d = lib.pa_paged_attention_decode_fp8
    dargs = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 2, 64, 8, 0.1, 1.0, 1.0, 4, 2, 128, 16, 0, None, 0, 0, None]

    def decode(**kw):
        a = list(dargs)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return d(*a)

    assert decode(a15=64) == 2               # FP8 pools hold head_dim 128 only
    assert decode(a11=float("nan")) == 1
    assert decode(a13=5) == 1                # q heads not a multiple of kv heads
    assert decode(a1=None) == 1
    assert decode(a7=0) == 0


def test_fp8_prefill_workspace_size(lib):
    # the 16-bit call's workspace, then [256 B header | chunk_seq | chunk_base |
    # table (B x max_blocks)], then K and V copy blocks of 16 rows x Hkv x D x 2 bytes
    B, T, Hq, Hkv, D, msl, mb = 4, 3000, 32, 8, 128, 4096, 256
    base = pa.prefill_workspace_bytes(B, T, Hq, D, msl)
    fixed = 256 + 2 * _align(B * 4) + _align(B * mb * 4)
    per = 2 * 16 * Hkv * D * 2
    chunks = min(B, T // 9)                  # at most one partial block per chunk
    for ckv in (0, 1, 16, 17, 5000):
        blocks = -(-ckv // 16) + chunks
        assert pa.prefill_fp8_workspace_bytes(B, T, Hq, Hkv, D, msl, mb, ckv) == base + fixed + blocks * per
    # never more copy blocks than the block tables can name
    assert pa.prefill_fp8_workspace_bytes(B, T, Hq, Hkv, D, msl, 2, 10**6) == \
        base + 256 + 2 * _align(B * 4) + _align(B * 2 * 4) + B * 2 * per
    assert pa.prefill_fp8_workspace_bytes(2, 10, 8, 8, 128, 64, 4, 32) == \
        pa.prefill_workspace_bytes(2, 10, 8, 128, 64) + 256 + 2 * _align(8) + _align(32) + (2 + 1) * 2 * 16 * 8 * 128 * 2
    assert pa.prefill_fp8_workspace_bytes(B, T, Hq, Hkv, D, msl, mb, -1) == 0
    assert pa.prefill_fp8_workspace_bytes(0, T, Hq, Hkv, D, msl, mb, 0) == 0


def test_fp8_prefill_rejects_a_workspace_without_copy_room(lib):
    # a chunk longer than 8 queries needs room for at least one copy block past
    # the 16-bit call's workspace and the copy's tables; checked before any CUDA call
    f = lib.pa_paged_attention_prefill_fp8
    B, T, Hq, Hkv, D, msl, mb = 2, 40, 8, 2, 128, 64, 4
    need = pa.prefill_fp8_workspace_bytes(B, T, Hq, Hkv, D, msl, mb, 0) - (T // 9 if T // 9 < B else B) * 2 * 16 * Hkv * D * 2
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, mb, FAKE, FAKE, B, T, 32, msl, 8, 0.1, 1.0, 1.0, Hq, Hkv, D, 16,
            FAKE, need + 2 * 16 * Hkv * D * 2 - 1, 0, None]
    assert f(*args) == 3                               # PA_ERR_WORKSPACE_TOO_SMALL


def test_gather_rejects_bad_arguments_on_the_host(lib):
    g = lib.pa_paged_kv_gather
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 64, 8, 2, 128, 2, None]

    def gather(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return g(*a)

    assert gather(a13=4) == 2                # element size
    assert gather(a12=8, a13=1) == 2         # a head-major FP8 row must be whole 16-byte chunks
    assert gather(a5=0) == 1 and gather(a0=None) == 1
    assert gather(a8=0) == 0


def test_noalloc_rejects_before_touching_the_device(lib):
    """The allocation-free decode checks its sizes against its fixed scratch
    before anything else, so these run without a GPU."""
    n = lib.pa_paged_attention_decode_noalloc
    # 64 heads x 1024 partitions of 16 tokens x (128 + 2) floats = 34 MB > 32 MiB
    assert n(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 1, 16 * 1024, 8, 0.1, 64, 8, 128, 16, 16, 1, None) == 3
    assert n(FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, -1, 64, 8, 0.1, 4, 2, 128, 16, 0, 1, None) == 1
    assert n(FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 1, -5, 8, 0.1, 4, 2, 128, 16, 0, 1, None) == 1
