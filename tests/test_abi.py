"""CPU checks of the C-ABI library: it builds, loads, exports every function include/gdn_decode.h
declares, agrees with the binding on struct layout, and rejects bad arguments on the host before
any CUDA call (so these run without a GPU: no call here reaches a launch)."""
import ctypes
import os
import re

import pytest

import ssm_recurrent_decode_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b((?:gdn|mamba)_\w+)\s*\(", text, re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in gdn.EXPORTS:
        assert n in names, n
    assert set(names) == set(gdn.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = gdn.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"{n} not exported"


def test_struct_layout_and_version():
    L = gdn.lib()
    assert L.gdn_abi_struct_size(0) == ctypes.sizeof(gdn.GdnStepArgs)
    assert L.gdn_abi_struct_size(1) == ctypes.sizeof(gdn.GdnRingArgs)
    assert L.gdn_abi_struct_size(2) == ctypes.sizeof(gdn.GdnFusedArgs)
    assert L.gdn_abi_struct_size(3) == ctypes.sizeof(gdn.GemvArgs)
    assert L.gdn_abi_struct_size(4) == ctypes.sizeof(gdn.GdnFrontArgs)
    assert L.gdn_abi_struct_size(5) == ctypes.sizeof(gdn.MambaArgs)
    assert L.gdn_abi_struct_size(9) == 0
    assert L.gdn_abi_version() == gdn.ABI_VERSION


def test_strerror():
    assert gdn.gdn_strerror(0) == "ok"
    assert "NULL" in gdn.gdn_strerror(-1)
    assert gdn.gdn_strerror(12345) == "unknown status"


def _valid_args():
    """Step arguments with fake, aligned, never dereferenced device addresses."""
    s = gdn.GdnStepArgs()
    s.B, s.H, s.HV, s.K, s.V, s.num_slots = 4, 2, 4, 128, 128, 4
    s.in_dtype, s.out_dtype = gdn.GDN_BF16, gdn.GDN_BF16
    base = 1 << 40
    s.q, s.k, s.v = base, base + 512, base + 1024
    s.q_stride = s.k_stride = s.v_stride = 2 * 2 * 128 + 4 * 128
    s.gate_mode = 0
    s.a, s.b, s.A_log, s.dt_bias = base + 4096, base + 8192, base + 12288, base + 16384
    s.state, s.out = base + (1 << 30), base + (1 << 31)
    return s


BAD = [
    ("null q", lambda s: setattr(s, "q", None), -1),
    ("null state", lambda s: setattr(s, "state", None), -1),
    ("null gate input", lambda s: setattr(s, "A_log", None), -1),
    ("K unsupported", lambda s: setattr(s, "K", 96), -2),
    ("V too large", lambda s: setattr(s, "V", 2048), -2),
    ("HV not a multiple of H", lambda s: setattr(s, "HV", 3), -2),
    ("num_slots below B", lambda s: setattr(s, "num_slots", 2), -2),
    ("negative B", lambda s: setattr(s, "B", -1), -2),
    ("bad dtype", lambda s: setattr(s, "in_dtype", 7), -3),
    ("q misaligned", lambda s: setattr(s, "q", (1 << 40) + 2), -4),
    ("k stride not a multiple of 4", lambda s: setattr(s, "k_stride", 1026), -4),
    ("state misaligned", lambda s: setattr(s, "state", (1 << 40) + 8), -4),
    ("row stride too short", lambda s: setattr(s, "v_stride", 100), -2),
    ("bad gate mode", lambda s: setattr(s, "gate_mode", 5), -6),
    ("direct gate without g", lambda s: setattr(s, "gate_mode", 1), -1),
]


@pytest.mark.parametrize("name,mutate,code", BAD, ids=[b[0] for b in BAD])
def test_step_rejects_bad_arguments_on_the_host(name, mutate, code):
    s = _valid_args()
    mutate(s)
    assert gdn.lib().gdn_decode_step(ctypes.byref(s), None) == code


def test_null_args_and_null_indices():
    L = gdn.lib()
    assert L.gdn_decode_step(None, None) == -1
    assert L.gdn_decode_fused(None, None) == -1
    s = _valid_args()
    assert L.gdn_decode_step_indexed(ctypes.byref(s), None, -1, None) == -1


def test_selftest_argument_checks():
    L = gdn.lib()
    assert L.gdn_selftest_bounded_wait(None, 1000, 0, None) == -1
    assert L.gdn_selftest_bounded_wait(1 << 40, 0, 0, None) == -6


def test_gemv_checks():
    L = gdn.lib()
    g = gdn.GemvArgs()
    assert L.gdn_gemv_bf16(None, None) == -1
    g.T, g.N, g.Kd, g.out_dtype = 2, 64, 100, 0          # Kd not a multiple of 8
    assert L.gdn_gemv_bf16(ctypes.byref(g), None) == -2
    g.Kd = 128
    assert L.gdn_gemv_bf16(ctypes.byref(g), None) == -1  # NULL pointers
    g.x, g.W, g.y, g.x_stride, g.y_stride = 1 << 40, 1 << 41, 1 << 42, 128, 64
    g.splits = 9                                       # more ranges than a cluster: a workspace
    assert L.gdn_gemv_bf16(ctypes.byref(g), None) == -1
    g.workspace, g.workspace_bytes = 1 << 43, 16
    assert L.gdn_gemv_bf16(ctypes.byref(g), None) == -2  # too small
    g.x = (1 << 40) + 8
    assert L.gdn_gemv_bf16(ctypes.byref(g), None) == -4
    assert L.gdn_gemv_workspace_bytes(2, 64, 9) == 9 * 2 * 64 * 4
    assert L.gdn_gemv_workspace_bytes(2, 64, 8) == 0     # up to 8 ranges add inside a cluster
    assert L.gdn_gemv_workspace_bytes(2, 64, 1) == 0
    for T, N, Kd in ((1, 17408, 5120), (8, 5120, 17408)):
        assert 1 <= L.gdn_gemv_default_splits(T, N, Kd) <= 8


def test_gemv_noalloc_checks_arguments_before_its_buffer_size():
    """gdn_gemv_bf16_noalloc returns gdn_gemv_bf16's codes for invalid calls, even when the
    request would also exceed its fixed buffer; GDN_ERR_SCRATCH only for valid calls that do. All
    of these return before any CUDA call."""
    L = gdn.lib()
    fn = L.gdn_gemv_bf16_noalloc
    g = gdn.GemvArgs()
    g.T, g.N, g.Kd, g.out_dtype = 8, 65536, 1024, 0     # 16 ranges: 8 Mi partial sums > 1 Mi
    g.x, g.W, g.y, g.x_stride, g.y_stride = 1 << 40, 1 << 41, 1 << 42, 1024, 65536
    g.splits = 65
    assert fn(ctypes.byref(g), None) == -2               # splits > 64: a shape error
    g.splits = -1
    assert fn(ctypes.byref(g), None) == -2
    g.splits = 16
    g.x = None
    assert fn(ctypes.byref(g), None) == -1               # a missing pointer
    g.x = (1 << 40) + 8
    assert fn(ctypes.byref(g), None) == -4               # misaligned x
    g.x = 1 << 40
    g.Kd = 1020
    assert fn(ctypes.byref(g), None) == -2               # Kd not a multiple of 8
    g.Kd = 1024
    assert fn(ctypes.byref(g), None) == -7               # valid, but larger than the buffer
    assert fn(None, None) == -1


def test_gemv_wait_limit_hook_round_trips():
    L = gdn.lib()
    before = L.gdn_gemv_set_wait_limit(0)
    assert before == 0
    assert L.gdn_gemv_set_wait_limit(4096) == 0
    assert L.gdn_gemv_set_wait_limit(-5) == 4096         # non-positive restores the default
    assert L.gdn_gemv_set_wait_limit(0) == 0


def test_empty_batch_launches_nothing():
    s = _valid_args()
    s.B = 0
    assert gdn.lib().gdn_decode_step(ctypes.byref(s), None) == 0


def test_buffered_ring_checks():
    L = gdn.lib()
    s = _valid_args()
    r = gdn.GdnRingArgs()
    r.L, r.ring_dtype = 0, gdn.GDN_BF16
    assert L.gdn_decode_buffered(ctypes.byref(s), None, -1, ctypes.byref(r), None) == -6
    r.L = 65
    assert L.gdn_decode_buffered(ctypes.byref(s), None, -1, ctypes.byref(r), None) == -6
    r.L = 8
    assert L.gdn_decode_buffered(ctypes.byref(s), None, -1, ctypes.byref(r), None) == -1
    assert L.gdn_decode_buffered(ctypes.byref(s), None, -1, None, None) == -1
    r.ring_dtype = 3
    assert L.gdn_decode_buffered(ctypes.byref(s), None, -1, ctypes.byref(r), None) == -3
    r.ring_dtype = gdn.GDN_BF16
    r.d_cache, r.k_cache, r.g_cache, r.write_pos = (1 << 41), (1 << 42), (1 << 43), (1 << 44)
    r.kernel = 7
    assert L.gdn_decode_buffered(ctypes.byref(s), None, -1, ctypes.byref(r), None) == -6


def test_fused_checks():
    L = gdn.lib()
    f = gdn.GdnFusedArgs()
    f.T, f.heads, f.head_dim, f.num_slots = 2, 4, 128, 4
    assert L.gdn_decode_fused(ctypes.byref(f), None) == -1          # NULL pointers
    f.head_dim = 100
    assert L.gdn_decode_fused(ctypes.byref(f), None) == -2
    f.head_dim, f.gate_kind = 128, 4
    assert L.gdn_decode_fused(ctypes.byref(f), None) == -6
    f.gate_kind, f.T = 0, 0
    assert L.gdn_decode_fused(ctypes.byref(f), None) == 0


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros((2, 2 * 2 * 16 + 4 * 16))
    q, k, v = gdn.split_mixed_qkv(x, 2, 4, 16, 16)
    with pytest.raises(TypeError, match="CUDA"):
        gdn.gdn_decode_step(q, k, v, torch.zeros((2, 4, 16, 16)), torch.zeros((2, 4, 16)), H=2,
                            a=torch.zeros(2, 4), b=torch.zeros(2, 4), A_log=torch.zeros(4),
                            dt_bias=torch.zeros(4))


def test_front_checks():
    """gdn_decode_front rejects bad arguments before launching anything."""
    L = gdn.lib()
    assert L.gdn_abi_struct_size(4) == ctypes.sizeof(gdn.GdnFrontArgs)
    assert L.gdn_front_proj_width(32, 128, gdn.GDN_FUSED_GATE_GDN) == 4 * 4096 + 64
    assert L.gdn_front_proj_width(16, 128, gdn.GDN_FUSED_GATE_KDA) == 5 * 2048 + 16
    assert L.gdn_front_proj_width(16, 128, 7) == 0
    assert L.gdn_decode_front(None, None) == -1
    a = gdn.GdnFrontArgs()
    a.T, a.hidden = 2, 5120
    a.core.heads, a.core.head_dim, a.core.num_slots = 32, 128, 4
    a.core.gate_kind = gdn.GDN_FUSED_GATE_GDN
    assert L.gdn_decode_front(ctypes.byref(a), None) == -1            # no z / o
    a.z, a.o = 1 << 40, (1 << 40) + 8
    assert L.gdn_decode_front(ctypes.byref(a), None) == -4            # o not 16-byte aligned
    a.o = 1 << 41
    assert L.gdn_decode_front(ctypes.byref(a), None) == -1            # no x, W, y (projection)
    a.in_splits = 9
    assert L.gdn_decode_front(ctypes.byref(a), None) == -6            # more ranges than a cluster
    a.in_splits, a.hidden = 0, 5121
    assert L.gdn_decode_front(ctypes.byref(a), None) == -2
    a.hidden, a.core.gate_kind = 5120, 5
    assert L.gdn_decode_front(ctypes.byref(a), None) == -6
    a.core.gate_kind, a.T = gdn.GDN_FUSED_GATE_GDN, 0
    assert L.gdn_decode_front(ctypes.byref(a), None) == 0             # nothing to do


@pytest.mark.parametrize("T,N,Kd,want", [
    (1, 17408, 5120, 1),    # 544 one-row CTAs fit the 608 slots (4 per SM) at one range
    (1, 5120, 17408, 2),    # one range would stage 34 KB of x per CTA (over 24 KB): two
    (8, 17408, 5120, 2),    # 136 tensor-core tiles; 272 CTAs fit the 456 slots (3 per SM), 544 do not
    (8, 5120, 17408, 8),    # 40 tiles: 320 CTAs at eight ranges still fit one wave
    (16, 5120, 17408, 8),
    (2, 4096, 1024, 2),     # at least 512 inputs per range caps the split count
])
def test_gemv_default_split_rule_on_the_page_shapes(T, N, Kd, want):
    """The split count for splits == 0: the largest power of two up to 8 whose grid fits one
    wave of resident CTAs (with its x slice staged), at least 512 inputs per range. Without a
    device the library takes GB300's counts (152 SMs; 4 one-row CTAs or 3 tensor-core CTAs per
    SM), and these are the counts measured at the Optimization Log's decode shapes."""
    import torch
    if torch.cuda.is_available():
        props = torch.cuda.get_device_properties(0)
        if props.multi_processor_count != 152:
            pytest.skip("the expected counts are GB300's")
    assert gdn.lib().gdn_gemv_default_splits(T, N, Kd) == want
