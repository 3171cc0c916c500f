"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every symbol the header declares, and its pure-host calls validate
arguments, report errors and persist the Fast-Run map."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from cnn_convolution_gemm_gb300 import build
    build.build()
    from cnn_convolution_gemm_gb300 import binding
    binding.load_library()
    return binding


def _header_functions():
    src = open(os.path.join(ROOT, "include", "gbconv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(conv_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported_and_bound(B):
    import ctypes
    names = _header_functions()
    assert len(names) >= 25
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B.SIGNATURES), set(names) ^ set(B.SIGNATURES)


def test_desc_validation(B):
    with pytest.raises(B.GbconvError) as e:
        B.conv_desc_create(1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 2, B.CONV_BF16)  # C % groups
    assert e.value.status_name == "CONV_ERR_BAD_PARAM"
    with pytest.raises(B.GbconvError):
        B.conv_desc_create(1, 4, 2, 2, 4, 5, 5, 1, 0, 1, 1, B.CONV_BF16)  # empty output
    d = B.conv_desc_create(2, 64, 56, 56, 64, 3, 3, 2, 1, 1, 1, B.CONV_BF16)
    assert B.conv_desc_get_output_dims(d) == (28, 28)
    with pytest.raises(B.GbconvError) as e:
        B.conv_desc_set_layout(d, B.CONV_NCHW)
    assert e.value.status_name == "CONV_ERR_UNSUPPORTED"
    B.conv_desc_destroy(d)


def test_size_limits_and_degenerate_shapes(B):
    # zero-sized dimensions are rejected at creation
    for dims in [(0, 8, 8, 8, 8), (1, 0, 8, 8, 8), (1, 8, 0, 8, 8), (1, 8, 8, 8, 0)]:
        N, C, H, W, K = dims
        with pytest.raises(B.GbconvError) as e:
            B.conv_desc_create(N, C, H, W, K, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
        assert e.value.status_name == "CONV_ERR_BAD_PARAM", dims
    # N*OH*OW at 2^31: the implicit GEMMs (32-bit GEMM row indices) step aside;
    # direct and Winograd (which runs chunks of images) still apply
    big = B.conv_desc_create(1 << 19, 64, 64, 64, 64, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    names = {n: ok for _, n, ok in (B.conv_algo_info(big, i) for i in range(B.CONV_ALGO_COUNT))}
    for n in ("igemm_tc_n64", "igemm_tc_n128", "igemm_tc_n256", "im2col_gemm"):
        assert not names[n], n
    assert names["direct"] and names["winograd_f2x2_3x3"]
    B.conv_desc_destroy(big)
    # just below: the implicit GEMM applies
    edge = B.conv_desc_create((1 << 19) - 1, 64, 64, 64, 64, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    assert B.conv_algo_info(edge, B.CONV_ALGO_IGEMM_N64)[2]
    B.conv_desc_destroy(edge)
    # a 1x1 output (kernel as large as the padded image) and a 1x1 kernel
    one = B.conv_desc_create(1, 8, 5, 5, 8, 5, 5, 1, 0, 1, 1, B.CONV_BF16)
    assert B.conv_desc_get_output_dims(one) == (1, 1)
    B.conv_desc_destroy(one)


def test_algo_table_and_applicability(B):
    d = B.conv_desc_create(32, 256, 56, 56, 256, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    infos = [B.conv_algo_info(d, i) for i in range(B.conv_algo_count(d))]
    names = {n: ok for _, n, ok in infos}
    assert names["direct"] and names["igemm_tc_n256"]
    dw = B.conv_desc_create(64, 144, 56, 56, 144, 3, 3, 1, 1, 1, 144, B.CONV_BF16)
    dnames = {n: ok for _, n, ok in (B.conv_algo_info(dw, i) for i in range(B.CONV_ALGO_COUNT))}
    assert not dnames["igemm_tc_n64"]  # grouped: implicit GEMM does not apply
    with pytest.raises(B.GbconvError) as e:
        B.conv_weights_packed_size(dw, B.CONV_ALGO_IGEMM_N64)
    assert e.value.status_name == "CONV_ERR_UNSUPPORTED"
    assert B.conv_weights_packed_size(d, B.CONV_ALGO_IGEMM_N128) == 256 * 9 * 256 * 2
    # C = 24 pads to one 64-channel block per filter tap
    e24 = B.conv_desc_create(64, 24, 56, 56, 144, 1, 1, 1, 0, 1, 1, B.CONV_BF16)
    assert B.conv_weights_packed_size(e24, B.CONV_ALGO_IGEMM_N64) == 144 * 64 * 2
    # the space-to-depth stem applies to stride-2 convs over 8 channels only
    stem = B.conv_desc_create(64, 8, 224, 224, 64, 7, 7, 2, 3, 1, 1, B.CONV_BF16)
    assert B.conv_algo_info(stem, B.CONV_ALGO_STEM_S2D)[2]
    assert B.conv_algo_info(stem, B.CONV_ALGO_STEM_S2D)[1] == "stem_s2d_igemm"
    assert B.conv_weights_packed_size(stem, B.CONV_ALGO_STEM_S2D) == 64 * 16 * 64 * 2
    assert B.conv_workspace_size(stem, B.CONV_ALGO_STEM_S2D) == 64 * 112 * 112 * 32 * 2
    assert not B.conv_algo_info(d, B.CONV_ALGO_STEM_S2D)[2]  # C = 256, stride 1
    odd = B.conv_desc_create(1, 8, 15, 16, 64, 7, 7, 2, 3, 1, 1, B.CONV_BF16)
    assert not B.conv_algo_info(odd, B.CONV_ALGO_STEM_S2D)[2]  # odd height
    # the space-to-depth-by-4 stem: 4 (or 8) channels, W % 32 == 0, K == 64;
    # 7x7 / 2 is a 3x3 conv over 4x4 blocks of 64 channels with 256 columns
    stem4 = B.conv_desc_create(64, 4, 224, 224, 64, 7, 7, 2, 3, 1, 1, B.CONV_BF16)
    assert B.conv_algo_info(stem4, B.CONV_ALGO_STEM_S2D4)[1:] == ("stem_s2d4_igemm", 1)
    assert B.conv_weights_packed_size(stem4, B.CONV_ALGO_STEM_S2D4) == 256 * 9 * 64 * 2
    assert B.conv_workspace_size(stem4, B.CONV_ALGO_STEM_S2D4) == 64 * 56 * 56 * 64 * 2
    assert not B.conv_algo_info(stem4, B.CONV_ALGO_STEM_S2D)[2]  # C = 4
    assert not B.conv_algo_info(stem4, B.CONV_ALGO_IGEMM_N64)[2]  # C % 8
    assert B.conv_algo_resolve(stem4) == B.CONV_ALGO_STEM_S2D4
    assert B.conv_algo_info(stem, B.CONV_ALGO_STEM_S2D4)[2]  # 8 channels: 128 per block
    assert B.conv_weights_packed_size(stem, B.CONV_ALGO_STEM_S2D4) == 256 * 9 * 128 * 2
    narrow_w = B.conv_desc_create(2, 4, 32, 48, 64, 7, 7, 2, 3, 1, 1, B.CONV_BF16)
    assert not B.conv_algo_info(narrow_w, B.CONV_ALGO_STEM_S2D4)[2]  # W % 32
    k32 = B.conv_desc_create(2, 4, 32, 32, 32, 7, 7, 2, 3, 1, 1, B.CONV_BF16)
    assert not B.conv_algo_info(k32, B.CONV_ALGO_STEM_S2D4)[2]  # K != 64
    for h in (d, dw, e24, stem, odd, stem4, narrow_w, k32):
        B.conv_desc_destroy(h)


def test_sm_pair_tile_applicability(B):
    """The 256 x 256 SM-pair implicit GEMM: bf16 NHWC, groups 1, C != 8 (the
    8-channel narrow mode stays single-SM), K > 128; same packed weights and no
    workspace."""
    def ok(*args, groups=1, dtype=None):
        d = B.conv_desc_create(*args, 1, groups, B.CONV_BF16 if dtype is None else dtype)
        try:
            r = B.conv_algo_info(d, B.CONV_ALGO_IGEMM_2SM)
            assert r[1] == "igemm_tc_2sm_n256"
            return r[2]
        finally:
            B.conv_desc_destroy(d)
    assert ok(32, 256, 56, 56, 256, 3, 3, 1, 1)
    assert ok(2, 64, 9, 9, 136, 1, 1, 2, 0)             # K just above one 128-wide tile
    assert not ok(2, 64, 9, 9, 128, 3, 3, 1, 1)         # K <= 128: a narrower tile
    assert not ok(2, 512, 7, 7, 512, 3, 3, 1, 1, groups=2)
    assert not ok(2, 8, 32, 32, 256, 7, 7, 2, 3)        # 8-channel stem input
    assert not ok(2, 64, 9, 9, 256, 3, 3, 1, 1, dtype=B.CONV_INT8)
    d = B.conv_desc_create(4, 256, 14, 14, 512, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    assert B.conv_weights_packed_size(d, B.CONV_ALGO_IGEMM_2SM) == B.conv_weights_packed_size(
        d, B.CONV_ALGO_IGEMM_N256)
    assert B.conv_workspace_size(d, B.CONV_ALGO_IGEMM_2SM) == 0
    B.conv_desc_destroy(d)


def test_fwd_argument_errors(B):
    d = B.conv_desc_create(1, 64, 8, 8, 64, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    with pytest.raises(B.GbconvError) as e:
        B.conv_fwd(d, 0, 0, 0, 0, 0, B.CONV_ALGO_DIRECT)
    assert e.value.status_name == "CONV_ERR_BAD_PARAM"
    with pytest.raises(B.GbconvError) as e:  # misaligned pointers are rejected before launch
        B.conv_fwd(d, 0x1008, 0x2000, 0, 0, 0x3000, B.CONV_ALGO_IGEMM_N64)
    assert e.value.status_name == "CONV_ERR_ALIGNMENT"
    with pytest.raises(B.GbconvError) as e:
        B.conv_fwd(d, 0x1000, 0x2000, 0, 0x4000, 0x3000, B.CONV_ALGO_IGEMM_N64)
    assert e.value.status_name == "CONV_ERR_BAD_PARAM"  # residual without has_residual
    B.conv_desc_destroy(d)


def test_fused_block_argument_errors(B):
    # the fused MobileNetV2 block validates shapes and pointers before any launch
    n = B.conv_mbv2_block_packed_size(24, 144, 24)
    assert n == 4 * 144 * 16 + 18 * 32 * 16 + 9 * 144 * 2  # [4][E][8] + [E/8][32][8] + [9][E]
    for bad in [(24, 192, 24), (32, 144, 24), (20, 144, 24), (24, 144, 36)]:
        with pytest.raises(B.GbconvError) as e:
            B.conv_mbv2_block_packed_size(*bad)
        assert e.value.status_name == "CONV_ERR_UNSUPPORTED"
    with pytest.raises(B.GbconvError) as e:
        B.conv_mbv2_block_fwd(1, 14, 14, 24, 144, 24, 0, 0x2000, 0, 0, False, 0x3000)
    assert e.value.status_name == "CONV_ERR_BAD_PARAM"  # NULL x
    with pytest.raises(B.GbconvError) as e:
        B.conv_mbv2_block_fwd(1, 14, 14, 16, 144, 24, 0x1000, 0x2000, 0, 0, True, 0x3000)
    assert e.value.status_name == "CONV_ERR_BAD_PARAM"  # residual needs C_in == C_out
    with pytest.raises(B.GbconvError) as e:
        B.conv_mbv2_block_fwd(1, 14, 14, 24, 144, 24, 0x1008, 0x2000, 0, 0, False, 0x3000)
    assert e.value.status_name == "CONV_ERR_ALIGNMENT"


def test_nc32hw32_layout_validation(B):
    # the blocked int8 layout: int8 only, C and K multiples of 32, groups 1
    bf = B.conv_desc_create(1, 64, 8, 8, 64, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    with pytest.raises(B.GbconvError) as e:
        B.conv_desc_set_layout(bf, B.CONV_NC32HW32)
    assert e.value.status_name == "CONV_ERR_UNSUPPORTED"
    i48 = B.conv_desc_create(1, 48, 8, 8, 64, 3, 3, 1, 1, 1, 1, B.CONV_INT8)
    with pytest.raises(B.GbconvError):
        B.conv_desc_set_layout(i48, B.CONV_NC32HW32)
    i64 = B.conv_desc_create(1, 64, 8, 8, 64, 3, 3, 1, 1, 1, 1, B.CONV_INT8)
    B.conv_desc_set_layout(i64, B.CONV_NC32HW32)
    B.conv_desc_set_requant(i64, 0x1000)  # a device address stand-in: no call runs here
    ok = {n: a for _, n, a in (B.conv_algo_info(i64, i) for i in range(B.CONV_ALGO_COUNT))}
    assert ok["int8_igemm_tc"] and ok["int8_igemm_tc_chunked"] and ok["direct"]
    assert not ok["int8_igemm_mma"]
    for h in (bf, i48, i64):
        B.conv_desc_destroy(h)


def test_input_shuffle_validation(B):
    d = B.conv_desc_create(1, 240, 28, 28, 240, 3, 3, 1, 1, 1, 240, B.CONV_BF16)
    with pytest.raises(B.GbconvError) as e:
        B.conv_desc_set_input_shuffle(d, 7)  # 7 does not divide 240
    assert e.value.status_name == "CONV_ERR_BAD_PARAM"
    B.conv_desc_set_input_shuffle(d, 3)
    ok = {n: a for _, n, a in (B.conv_algo_info(d, i) for i in range(B.CONV_ALGO_COUNT))}
    assert ok["depthwise3x3"] and ok["direct"]
    assert not any(a for n, a in ok.items() if n not in ("depthwise3x3", "direct"))
    g = B.conv_desc_create(1, 64, 8, 8, 64, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    B.conv_desc_set_input_shuffle(g, 4)
    assert not B.conv_algo_info(g, B.CONV_ALGO_IGEMM_N64)[2]
    B.conv_desc_set_input_shuffle(g, 1)  # off again
    assert B.conv_algo_info(g, B.CONV_ALGO_IGEMM_N64)[2]
    for h in (d, g):
        B.conv_desc_destroy(h)


def test_selftest_argument_checks(B):
    for bad in (0, 10_000_001):
        with pytest.raises(B.GbconvError) as e:
            B.conv_selftest_wait_timeout(bad, None)
        assert e.value.status_name == "CONV_ERR_BAD_PARAM"


def test_status_strings(B):
    assert B.conv_status_string(0) == "CONV_OK"
    assert B.conv_status_string(6) == "CONV_ERR_TIMEOUT"
    assert B.conv_version().startswith("gbconv")


def test_fwd_host_scratch_and_argument_errors(B):
    # scratch = 2 x (input chunk + output chunk) + the chunk's workspace, each 256-rounded
    d = B.conv_desc_create(8, 64, 10, 10, 128, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    xi, yi = 64 * 100 * 2, 128 * 100 * 2
    r256 = lambda b: (b + 255) // 256 * 256
    assert B.conv_fwd_host_scratch_size(d, B.CONV_ALGO_IGEMM_N128, 3) == 2 * (
        r256(3 * xi) + r256(3 * yi))
    assert B.conv_fwd_host_scratch_size(d, B.CONV_ALGO_IGEMM_N128, 0) == 2 * (8 * xi + 8 * yi)
    assert B.conv_fwd_host_scratch_size(d, B.CONV_ALGO_IGEMM_N128, 99) == 2 * (8 * xi + 8 * yi)
    n0 = B.conv_launch_count()
    for args, status in [
        ((d, 0, 16, None, None, 16, 2, 2, 256, 1 << 20, None), "CONV_ERR_BAD_PARAM"),  # NULL x
        ((d, 16, 16, None, 16, 16, 2, 2, 256, 1 << 20, None), "CONV_ERR_BAD_PARAM"),  # residual
        ((d, 16, 16, None, None, 16, 2, 2, 272, 1 << 20, None), "CONV_ERR_ALIGNMENT"),  # scratch
        ((d, 16, 16, None, None, 16, 2, 2, 256, 1024, None), "CONV_ERR_WORKSPACE"),
    ]:
        with pytest.raises(B.GbconvError) as e:
            B.conv_fwd_host(*args)
        assert e.value.status_name == status
    assert B.conv_launch_count() == n0
    B.conv_desc_destroy(d)


def test_launch_counter_does_not_move_on_rejected_calls(B):
    # calls that fail validation on the host launch nothing
    n0 = B.conv_launch_count()
    h = B.conv_desc_create(2, 64, 8, 8, 64, 3, 3, 1, 1)
    try:
        with pytest.raises(B.GbconvError):
            B.conv_fwd(h, 0, 0, None, None, 0, B.CONV_ALGO_IGEMM_N64, None, 0, None)
    finally:
        B.conv_desc_destroy(h)
    assert B.conv_launch_count() == n0


def test_fastrun_file_roundtrip_and_corruption(B, tmp_path):
    B.conv_fastrun_clear()
    p = tmp_path / "map.txt"
    B.conv_fastrun_save(str(p))
    text = p.read_text()
    assert "version" in text and "end 0" in text
    B.conv_fastrun_load(str(p))
    bad = tmp_path / "bad.txt"
    bad.write_text(text.replace("end 0", "end 3"))
    with pytest.raises(B.GbconvError) as e:
        B.conv_fastrun_load(str(bad))
    assert e.value.status_name == "CONV_ERR_FASTRUN_FILE"
    bad.write_text("garbage\n")
    with pytest.raises(B.GbconvError):
        B.conv_fastrun_load(str(bad))
    with pytest.raises(B.GbconvError):
        B.conv_fastrun_load(str(tmp_path / "missing.txt"))
    d = B.conv_desc_create(1, 8, 4, 4, 8, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    with pytest.raises(B.GbconvError) as e:
        B.conv_fastrun_lookup(d)
    assert e.value.status_name == "CONV_ERR_NOT_FOUND"
    B.conv_desc_destroy(d)


def test_fastrun_log_and_map_file_environment(B, tmp_path):
    """GBCONV_FASTRUN_FILE loads the map before the first lookup and GBCONV_LOG=1
    reports the load and each resolution on stderr (a fresh process: both
    variables are read once)."""
    import subprocess
    import sys
    import textwrap
    from cnn_convolution_gemm_gb300 import binding
    version = binding.conv_version()
    key = "N1_C64_H8_W8_K64_R3_S3_st1_p1_d1_g1_t0_l0_a0_r0_q0"
    p = tmp_path / "map.txt"
    p.write_text(f"version {version}\nentry nodevice {key} direct\nend 1\n")
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        from cnn_convolution_gemm_gb300 import binding as B
        d = B.conv_desc_create(1, 64, 8, 8, 64, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
        print(B.conv_algo_resolve(d))
        d2 = B.conv_desc_create(1, 64, 8, 8, 128, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
        print(B.conv_algo_resolve(d2))
    """)
    env = dict(os.environ, GBCONV_LOG="1", GBCONV_FASTRUN_FILE=str(p))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[gbconv]")]
    load = [ln for ln in lines if "fastrun load" in ln]
    assert len(load) == 1 and str(p) in load[0], lines
    resolved = [ln for ln in lines if ln.startswith("[gbconv] resolve")]
    assert len(resolved) == 2, lines
    if "1 entries for nodevice" in load[0]:  # no GPU: the entry is this machine's
        assert resolved[0] == f"[gbconv] resolve {key} -> direct (fastrun map)"
        assert r.stdout.split()[0] == str(B.CONV_ALGO_DIRECT)
    else:  # an entry for another device is skipped
        assert "(heuristic)" in resolved[0]
    assert resolved[1].endswith("-> igemm_tc_n128 (heuristic)"), resolved
