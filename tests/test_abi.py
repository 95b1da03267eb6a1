"""The C ABI without a GPU: the library loads, exports every function the
header declares, reports sizes and stage names, and rejects bad arguments on
the host before any CUDA call."""
import ctypes

import pytest

from state_space_model_09_b300 import ssd as S


def test_exports_every_declared_function():
    names = S.header_functions()
    assert {"ssd_fwd", "ssd_multistep", "ssd_fwd_workspace_size", "ssd_status_string",
            "ssd_version", "ssd_fwd_profiled", "ssd_check_device_error"} <= set(names)
    lib = S.library_handle()
    for n in names:
        assert getattr(lib, n) is not None, n


def test_version_and_status_strings():
    assert S.ssd_version() == 10000
    for st in range(5):
        assert S.ssd_status_string(st)
    assert S.ssd_status_string(99) == "unknown status"


def _dims(**kw):
    base = dict(batch=8, seqlen=2048, nheads=80, headdim=64, dstate=128, ngroups_b=1,
                ngroups_c=1, io_dtype=S.SSD_BF16, dt_softplus=True)
    base.update(kw)
    return S.make_dims(**base)


def test_workspace_size_layout():
    d = _dims()
    nc = 8
    cs = 8 * 80 * nc * 256 * 4
    st = 8 * nc * 80 * 128 * 64
    # tensor-core path: the bf16 chunk initial states; one (B, C) group with
    # 256-token chunks of 64-wide heads adds one byte per (batch, chunk, head)
    # (whether the head-pair chunk scan takes that unit) and the per-token
    # log2 decays [b, H, T] in float32.  Its 320 (batch, head pair) chunk-state
    # items fill two waves of 148 SMs and 24 more: those 24 (batch 7, heads
    # 32-79) run in four segments of two chunks, whose hand-off takes each
    # segment's final state and decay and each chunk's decay product
    rows, nseg = 48, 4
    handoff = rows * nseg * 128 * 64 * 4 + rows * nseg * 4 + rows * nc * 4
    assert S.ssd_fwd_workspace_size(d, 256) == \
        st * 2 + handoff + 8 * nc * 80 + 8 * 80 * 2048 * 4
    d_g2 = _dims(ngroups_b=2, ngroups_c=2)
    assert S.ssd_fwd_workspace_size(d_g2, 256) == st * 2
    # float32 path: cumsums, chunk states and chunk initial states in float32
    d32 = _dims(io_dtype=S.SSD_F32)
    assert S.ssd_fwd_workspace_size(d32, 256) == cs + st * 4 + st * 4
    # ragged T: ceil(T / Q) chunks
    d2 = _dims(seqlen=2049)
    assert S.ssd_fwd_workspace_size(d2, 256) > S.ssd_fwd_workspace_size(d, 256)


def test_stage_names_follow_the_path(monkeypatch):
    monkeypatch.delenv("SSD_FUSED", raising=False)
    monkeypatch.delenv("SSD_CHUNK_SCAN", raising=False)
    names = lambda d, q=256: [S.ssd_fwd_stage_name(d, q, i) for i in range(S.ssd_fwd_num_stages(d, q))]
    # 256-token chunks of 64-wide heads, one (B, C) group: the one-pass kernel;
    # the last wave's items split into segments need its prepass
    assert names(_dims()) == ["chunk_fused_prepass", "chunk_fused_hb", "chunk_scan_flagged"]
    # 37 x 40 head pairs = ten full waves of 148: no split, no prepass
    assert names(_dims(batch=37)) == ["chunk_fused_hb", "chunk_scan_flagged"]
    # one long sequence over 80 heads: 40 items, fewer than the SMs, so the
    # two-pass kernels (the one-pass kernel on request)
    long = _dims(batch=1, seqlen=16384)
    assert names(long) == ["dt_decay", "chunk_state_hb", "state_fixup", "chunk_scan_hb"]
    assert S.ssd_fwd_workspace_size(long, 256) > 1 * 64 * 80 * 128 * 64 * 2
    monkeypatch.setenv("SSD_FUSED", "1")
    assert names(long) == ["chunk_fused_prepass", "chunk_fused_hb", "chunk_scan_flagged"]
    monkeypatch.delenv("SSD_FUSED")
    assert names(_dims(ngroups_c=2)) == ["chunk_state_pass_tc", "chunk_scan_hl"]
    # the hybrid shape (128-token chunks of 128-wide heads, grouped B and C):
    # 4 x 32 one-head items fill more than half the SMs -> the one-pass kernel
    hyb = _dims(batch=4, seqlen=4096, nheads=32, headdim=128, ngroups_b=8, ngroups_c=32)
    assert names(hyb, 128) == ["chunk_fused_hb", "chunk_scan_flagged"]
    # one batch row: 32 items, too few -> the two-pass kernels
    assert "chunk_fused_hb" not in names(_dims(batch=1, seqlen=4096, nheads=32, headdim=128,
                                               ngroups_b=8, ngroups_c=32), 128)
    assert names(_dims(io_dtype=S.SSD_F32), 64) == \
        ["dt_cumsum", "chunk_state_simt", "state_passing", "chunk_scan_simt"]
    assert names(_dims(headdim=128), 128)[-2:] == ["chunk_fused_hb", "chunk_scan_flagged"]
    assert names(_dims(headdim=128, batch=1, nheads=32), 128)[-1] == "chunk_scan_hl"
    assert S.ssd_fwd_stage_name(_dims(), 256, 3) is None
    assert S.ssd_fwd_num_stages(_dims(), 128) == 2
    assert S.ssd_fwd_num_stages(_dims(io_dtype=S.SSD_F32), 256) == 4
    # SSD_FUSED=0: the two-pass head-pair kernels; the last wave's chunk-state
    # items split into segments joined by a fix-up stage
    monkeypatch.setenv("SSD_FUSED", "0")
    assert names(_dims()) == ["dt_decay", "chunk_state_hb", "state_fixup", "chunk_scan_hb"]
    assert names(_dims(batch=37)) == ["dt_decay", "chunk_state_hb", "chunk_scan_hb"]
    assert names(long) == ["dt_decay", "chunk_state_hb", "state_fixup", "chunk_scan_hb"]


def _scan_stage(d, chunk=256):
    return S.ssd_fwd_stage_name(d, chunk, S.ssd_fwd_num_stages(d, chunk) - 1)


def test_chunk_scan_form_follows_work_per_cta_and_override(monkeypatch):
    monkeypatch.delenv("SSD_CHUNK_SCAN", raising=False)
    monkeypatch.setenv("SSD_FUSED", "0")  # the two-pass kernels choose a chunk-scan form
    d = _dims()  # 64 (batch, chunk) items x 40 head pairs: head pairs
    window = _dims(batch=1, seqlen=4096)  # 16 items: too few pairs per CTA
    assert _scan_stage(d) == "chunk_scan_hb"
    assert _scan_stage(window) == "chunk_scan_hl"
    sizes = (S.ssd_fwd_workspace_size(d, 256), S.ssd_fwd_workspace_size(window, 256))
    monkeypatch.setenv("SSD_CHUNK_SCAN", "head")
    assert _scan_stage(d) == "chunk_scan_hl"
    monkeypatch.setenv("SSD_CHUNK_SCAN", "pair")
    assert _scan_stage(window) == "chunk_scan_hb"
    # the workspace (with the decay-range flags) does not depend on the choice
    assert (S.ssd_fwd_workspace_size(d, 256), S.ssd_fwd_workspace_size(window, 256)) == sizes


@pytest.mark.parametrize("kw,chunk,status", [
    (dict(headdim=24), 256, S.SSD_ERR_UNSUPPORTED),
    (dict(dstate=272), 256, S.SSD_ERR_UNSUPPORTED),
    (dict(ngroups_b=3), 256, S.SSD_ERR_INVALID_ARG),
    (dict(batch=0), 256, S.SSD_ERR_INVALID_ARG),
    (dict(io_dtype=7), 256, S.SSD_ERR_INVALID_ARG),
    (dict(), 96, S.SSD_ERR_UNSUPPORTED),
])
def test_bad_dims_rejected_on_host(kw, chunk, status):
    d = _dims(**kw)
    assert S.ssd_fwd_workspace_size(d, chunk) == 0
    lib = S.library_handle()
    # fake, aligned, non-null "device" pointers: validation fails before any use
    p = ctypes.c_void_p(1 << 20)
    r = lib.ssd_fwd(ctypes.byref(d), p, p, p, p, p, None, None, chunk, ctypes.c_void_p(2 << 20),
                    None, ctypes.c_void_p(3 << 20), 1 << 40, None)
    assert r == status


def test_null_and_misaligned_pointers_rejected():
    d = _dims()
    lib = S.library_handle()
    good = [ctypes.c_void_p((k + 1) << 32) for k in range(5)]
    y, ws = ctypes.c_void_p(9 << 32), ctypes.c_void_p(10 << 32)
    args = lambda ins, yy: [ctypes.byref(d)] + ins + [None, None, 256, yy, None, ws, 1 << 40, None]
    assert lib.ssd_fwd(*args([None] + good[1:], y)) == S.SSD_ERR_INVALID_ARG
    assert lib.ssd_fwd(*args(good, ctypes.c_void_p((9 << 32) + 8))) == S.SSD_ERR_INVALID_ARG
    # short workspace
    r = lib.ssd_fwd(ctypes.byref(d), *good, None, None, 256, y, None, ws, 1024, None)
    assert r == S.SSD_ERR_INVALID_ARG
    # output aliasing an input
    r = lib.ssd_fwd(ctypes.byref(d), *good, None, None, 256, good[0], None, ws, 1 << 40, None)
    assert r == S.SSD_ERR_INVALID_ARG


def test_multistep_validation():
    lib = S.library_handle()
    d = _dims(seqlen=17)
    p = [ctypes.c_void_p((k + 1) << 32) for k in range(11)]
    assert lib.ssd_multistep(ctypes.byref(d), *p, None) == S.SSD_ERR_UNSUPPORTED
    d = _dims(seqlen=8)
    q = list(p)
    q[7] = None  # j
    assert lib.ssd_multistep(ctypes.byref(d), *q, None) == S.SSD_ERR_INVALID_ARG
    q = list(p)
    q[9] = q[6]  # h_j aliases h_cache
    assert lib.ssd_multistep(ctypes.byref(d), *q, None) == S.SSD_ERR_INVALID_ARG


def test_sequential_workspace_is_independent_of_the_prompt_length():
    w = S.ssd_fwd_sequential_workspace_size
    short, long = _dims(batch=1, seqlen=1000), _dims(batch=1, seqlen=1_000_000)
    assert w(short, 256, 512) == w(long, 256, 512) > 0
    # batch > 1 adds a staging copy of one window of x, dt, B, C and y
    assert w(_dims(batch=2, seqlen=1000), 256, 512) > w(_dims(batch=1, seqlen=1000), 256, 512)
    # a window no longer than the sequence is what is planned for
    assert w(short, 256, 10_000) == w(short, 256, 1000)
    assert w(short, 256, 0) == 0 and w(short, 96, 512) == 0


def test_sequential_rejects_bad_arguments_on_host():
    d = _dims(batch=1, seqlen=1000)
    n = S.ssd_fwd_sequential_workspace_size(d, 256, 256)
    lib = S.library_handle()
    fake = ctypes.c_void_p(0x10000)
    args = [ctypes.byref(d)] + [fake] * 7 + [256, 256, fake, fake, fake]
    # workspace too small, window 0, NULL x
    assert lib.ssd_fwd_sequential(*args, n - 1, None) == S.SSD_ERR_INVALID_ARG
    a2 = list(args); a2[9] = 0
    assert lib.ssd_fwd_sequential(*a2, n, None) == S.SSD_ERR_INVALID_ARG
    a3 = list(args); a3[1] = None
    assert lib.ssd_fwd_sequential(*a3, n, None) == S.SSD_ERR_INVALID_ARG


def test_sequential_checks_every_buffer_before_the_first_window():
    """Aliasing and misalignment anywhere in the whole tensors are reported
    before any window is enqueued (fake, never dereferenced pointers)."""
    d = _dims(batch=1, seqlen=1000)
    n = S.ssd_fwd_sequential_workspace_size(d, 256, 256)
    lib = S.library_handle()
    # x dt A B C D h0 | y h_final workspace: distinct, far apart, 16-byte aligned
    ptr = [ctypes.c_void_p((i + 1) << 34) for i in range(10)]

    def call(p):
        return lib.ssd_fwd_sequential(ctypes.byref(d), *p[:7], 256, 256, *p[7:], n, None)

    alias = list(ptr)
    alias[7] = alias[0]                      # y aliases x
    assert call(alias) == S.SSD_ERR_INVALID_ARG
    tail = list(ptr)
    tail[8] = ctypes.c_void_p(ptr[0].value + 64)  # h_final inside x
    assert call(tail) == S.SSD_ERR_INVALID_ARG
    odd = list(ptr)
    odd[1] = ctypes.c_void_p(ptr[1].value + 8)    # dt off the 16-byte boundary
    assert call(odd) == S.SSD_ERR_INVALID_ARG
    ws_in = list(ptr)
    ws_in[9] = ctypes.c_void_p(ptr[3].value + 16)  # workspace overlapping B
    assert call(ws_in) == S.SSD_ERR_INVALID_ARG


def test_sequential_stages_dt_windows_that_would_break_alignment():
    """Batch 1 with H = 3: a 250-token window starts 3000 bytes into dt, off
    the 16-byte boundary, so dt windows are staged (more workspace); with a
    window that keeps the boundary (256 x 3 x 4 bytes) nothing is staged."""
    w = S.ssd_fwd_sequential_workspace_size
    d = _dims(batch=1, seqlen=1000, nheads=3, ngroups_b=1, ngroups_c=1)
    d256 = w(d, 256, 256)
    d250 = w(d, 256, 250)
    assert d250 > 0 and d256 > 0
    fwd250 = S.ssd_fwd_workspace_size(_dims(batch=1, seqlen=250, nheads=3, ngroups_b=1,
                                            ngroups_c=1), 256)
    fwd256 = S.ssd_fwd_workspace_size(_dims(batch=1, seqlen=256, nheads=3, ngroups_b=1,
                                            ngroups_c=1), 256)
    assert d250 - fwd250 > d256 - fwd256


def test_cp_calls_reject_bad_arguments_on_host():
    """Context-parallel calls: rank outside 0..nranks-1, NULL or misaligned
    pointers and aliasing are reported before anything is launched (fake,
    never dereferenced pointers)."""
    lib = S.library_handle()
    d = _dims(batch=2, seqlen=1000)
    n = S.ssd_cp_workspace_size(d)
    assert n >= 2 * 1000 * 80 * 4 + 2 * 80 * 128 * 64 * 4
    assert S.ssd_cp_workspace_size(_dims(headdim=24)) == 0
    # decays finals dt A C y h_final workspace
    ptr = [ctypes.c_void_p((i + 1) << 36) for i in range(8)]

    def correct(nranks, rank, p, ws=n):
        return lib.ssd_cp_correct(ctypes.byref(d), nranks, rank, *p[:7], p[7], ws, None)

    assert correct(2, 2, ptr) == S.SSD_ERR_INVALID_ARG      # rank >= nranks
    assert correct(2, -1, ptr) == S.SSD_ERR_INVALID_ARG     # rank < 0
    assert correct(0, 0, ptr) == S.SSD_ERR_INVALID_ARG      # no ranks
    assert correct(2, 1, ptr, n - 1) == S.SSD_ERR_INVALID_ARG  # short workspace
    alias = list(ptr); alias[5] = alias[4]                   # y aliases C
    assert correct(2, 1, alias) == S.SSD_ERR_INVALID_ARG
    alias = list(ptr); alias[6] = ctypes.c_void_p(ptr[1].value + 256)  # h_final inside finals
    assert correct(2, 1, alias) == S.SSD_ERR_INVALID_ARG
    odd = list(ptr); odd[2] = ctypes.c_void_p(ptr[2].value + 4)
    assert correct(2, 1, odd) == S.SSD_ERR_INVALID_ARG      # dt misaligned
    null = list(ptr); null[4] = None
    assert correct(2, 1, null) == S.SSD_ERR_INVALID_ARG     # NULL C
    # segment decay: dt A decay workspace
    dec = [ctypes.c_void_p((i + 1) << 36) for i in range(4)]
    seg = lambda p, ws=n: lib.ssd_cp_segment_decay(ctypes.byref(d), *p, ws, None)
    assert seg(dec, 16) == S.SSD_ERR_INVALID_ARG            # short workspace
    alias = list(dec); alias[2] = alias[0]                   # decay aliases dt
    assert seg(alias) == S.SSD_ERR_INVALID_ARG


def test_verify_rejects_bad_arguments_on_host():
    """Host-side checks only: every case returns before anything touches the
    (fake, never dereferenced) device pointers."""
    lib = S.library_handle()
    d = _dims(batch=2, seqlen=8)
    # 13 distinct, far-apart, 16-byte-aligned addresses for:
    # x_prev dt_prev B_prev j_prev x dt A B C D h_cache y h_next
    ptr = [ctypes.c_void_p((i + 1) << 32) for i in range(13)]

    def call(dims, k_prev, p):
        return lib.ssd_verify(ctypes.byref(dims), k_prev, *p, None)

    no_prev = list(ptr)
    no_prev[0] = None
    assert call(d, 8, no_prev) == S.SSD_ERR_INVALID_ARG           # NULL previous drafts
    assert call(_dims(batch=2, seqlen=17), 8, ptr) == S.SSD_ERR_UNSUPPORTED   # K > 16
    assert call(d, 17, ptr) == S.SSD_ERR_UNSUPPORTED              # k_prev > 16
    assert call(d, 0, ptr) == S.SSD_ERR_INVALID_ARG               # k_prev < 1
    alias = list(ptr)
    alias[12] = alias[10]
    assert call(d, 8, alias) == S.SSD_ERR_INVALID_ARG             # h_next aliases h_cache
    odd = list(ptr)
    odd[4] = ctypes.c_void_p(ptr[4].value + 8)
    assert call(d, 8, odd) == S.SSD_ERR_INVALID_ARG               # x not 16-byte aligned
