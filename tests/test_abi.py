"""Host-side checks of the C ABI: the library loads, exports what the header
declares, and rejects bad arguments before touching the device (no GPU
needed: every call here returns before any CUDA work)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(REPO, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(moe_w4a8_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib(cuda_lib):
    from bit_moe_expert_router_gb300 import binding
    return binding._load()


def test_header_declares_the_entry_points():
    names = _declared_symbols()
    assert {"moe_w4a8_forward", "moe_w4a8_route", "moe_w4a8_workspace_size", "moe_w4a8_version",
            "moe_w4a8_status_string", "moe_w4a8_gemm1_partials", "moe_w4a8_gemm2_partials",
            "moe_w4a8_forward_debug", "moe_w4a8_device_status", "moe_w4a8_forward_host",
            "moe_w4a8_forward_host_workspace_size", "moe_w4a8_forward_bf16", "moe_w4a8_forward_w2w4",
            "moe_w4a8_forward_bf16_workspace_size", "moe_w4a8_debug_routing", "moe_w4a8_forward_routed"} <= names


def test_library_exports_every_declared_symbol(cuda_lib, lib):
    out = subprocess.run(["nm", "-D", "--defined-only", cuda_lib], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (moe_w4a8_\w+)", out))
    missing = _declared_symbols() - exported
    assert not missing, missing
    for name in _declared_symbols():
        assert getattr(lib, name) is not None
    # nothing but the C ABI is exported
    assert all(s.startswith("moe_w4a8_") for s in re.findall(r"\bT (\w+)", out))


def test_version_and_status_strings(lib):
    from bit_moe_expert_router_gb300 import binding
    assert lib.moe_w4a8_version() == binding.ABI_VERSION == 4
    for s in range(6):
        assert binding.moe_w4a8_status_string(s)
    assert binding.moe_w4a8_status_string(99) == "unknown status"


def test_workspace_size_grows_with_tokens(lib):
    from bit_moe_expert_router_gb300 import binding
    from bit_moe_expert_router_gb300.synth import WORKLOADS
    w = WORKLOADS["decode_t4"]
    sizes = [binding.moe_w4a8_workspace_size(binding.dims_of(T, w.H, w.I, w.E, w.S, w.top_k, w.group))
             for T in (1, 4, 64, 8192)]
    assert all(s % 256 == 0 for s in sizes)
    assert sizes == sorted(sizes) and sizes[0] < sizes[-1]
    # the per-pair intermediates dominate: h (I floats) and Y (H floats) per pair row
    P = 8192 * (w.top_k + w.S)
    assert sizes[-1] >= P * (w.I + w.H) * 4


@pytest.mark.parametrize("field,value,status", [
    ("E", 0, 1), ("top_k", 0, 1), ("top_k", 9, 1), ("group", 48, 1), ("group", 0, 1), ("H", 200, 1),
    ("I", 96, 1), ("T", -1, 1), ("n_shared", -1, 1),
    ("E", 2048, 2), ("group", 512, 1), ("n_shared", 9, 2), ("H", 320, 2),
    ("H", 1 << 17, 2), ("I", 1 << 17, 2), ("H", 1 << 40, 2),
])
def test_bad_dims_are_rejected(lib, field, value, status):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(16, 256, 128, 8, 0, 2, 64)
    setattr(d, field, value)
    assert lib.moe_w4a8_workspace_size(ctypes.byref(d)) == 0
    rc = lib.moe_w4a8_forward(None, None, None, None, None, None, None, ctypes.byref(d), None, None, 0, None)
    assert rc == status


def test_partials_workspace_size_follows_the_pair_limit(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(16, 256, 128, 8, 0, 2, 64)
    assert lib.moe_w4a8_partials_workspace_size(ctypes.byref(d), ctypes.c_int64(0)) > 0
    assert lib.moe_w4a8_partials_workspace_size(ctypes.byref(d), ctypes.c_int64((1 << 24) - 1)) > 0
    assert lib.moe_w4a8_partials_workspace_size(ctypes.byref(d), ctypes.c_int64(1 << 24)) == 0
    assert lib.moe_w4a8_partials_workspace_size(ctypes.byref(d), ctypes.c_int64(-1)) == 0


def test_group_beyond_limit_is_unsupported(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(16, 1024, 512, 8, 0, 2, 512)
    assert lib.moe_w4a8_forward(None, None, None, None, None, None, None, ctypes.byref(d), None, None, 0, None) == 2


def test_null_and_misaligned_pointers_are_rejected(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(16, 256, 128, 8, 0, 2, 64)
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: the checks fail first
    odd = ctypes.c_void_p(0x100008)
    args = [fake] * 7
    assert lib.moe_w4a8_forward(*args[:3], None, *args[4:7], ctypes.byref(d), fake, fake, 1 << 30, None) == 1
    assert lib.moe_w4a8_forward(*args[:3], odd, *args[4:7], ctypes.byref(d), fake, fake, 1 << 30, None) == 1
    # workspace: misaligned, then too small
    ws_unaligned = ctypes.c_void_p(0x100010)
    assert lib.moe_w4a8_forward(*args, ctypes.byref(d), fake, ws_unaligned, 1 << 30, None) == 1
    need = lib.moe_w4a8_workspace_size(ctypes.byref(d))
    assert lib.moe_w4a8_forward(*args, ctypes.byref(d), fake, fake, need - 256, None) == 3
    assert lib.moe_w4a8_route(fake, ctypes.byref(d), fake, fake, fake, fake, fake, None, fake, need, None) == 1
    # the routing read-back: a null output, then a workspace too small
    assert lib.moe_w4a8_debug_routing(ctypes.byref(d), fake, need, fake, None, fake, fake, None) == 1
    assert lib.moe_w4a8_debug_routing(ctypes.byref(d), fake, need - 256, fake, fake, fake, fake, None) == 3
    # the routed layer: no routing, then a misaligned weight array, then a workspace too small
    assert lib.moe_w4a8_forward_routed(fake, fake, None, fake, *([fake] * 4), ctypes.byref(d), fake, fake, need,
                                       None) == 1
    assert lib.moe_w4a8_forward_routed(fake, fake, fake, odd, *([fake] * 4), ctypes.byref(d), fake, fake, need,
                                       None) == 1
    assert lib.moe_w4a8_forward_routed(fake, fake, fake, fake, *([fake] * 4), ctypes.byref(d), fake, fake,
                                       need - 256, None) == 3


def test_partials_workspace_covers_grouping_and_fp16_rows(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(64, 2048, 512, 512, 1, 10, 128)
    small, big = (binding.moe_w4a8_partials_workspace_size(d, n) for n in (8, 4096))
    assert small % 256 == 0 and small < big
    # the fp16 activation rows and down-projection rows of the n_pairs pairs
    assert small >= 2 * 8 * d.H + 2 * 8 * d.I
    assert big >= 4096 * (d.I + d.H) * 4 + 2 * 4096 * d.I
    assert lib.moe_w4a8_partials_workspace_size(ctypes.byref(d), -1) == 0
    d.group = 48
    assert lib.moe_w4a8_partials_workspace_size(ctypes.byref(d), 8) == 0


def test_empty_batch_is_a_no_op(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(0, 256, 128, 8, 0, 2, 64)
    fake = ctypes.c_void_p(0x100000)
    # T = 0: valid, nothing enqueued, activations may be null
    assert lib.moe_w4a8_forward(None, None, None, fake, fake, fake, fake, ctypes.byref(d), None, None, 0, None) == 0
    assert lib.moe_w4a8_route(None, ctypes.byref(d), None, None, None, None, None, None, None, 0, None) == 0


def test_engine_and_status_arguments_are_checked(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(4, 2048, 512, 512, 1, 10, 128)
    fake = ctypes.c_void_p(0x100000)
    need = lib.moe_w4a8_workspace_size(ctypes.byref(d))
    # an engine outside {-1, 0, 1, 2} is rejected before anything is enqueued
    assert lib.moe_w4a8_forward_debug(*[fake] * 7, ctypes.byref(d), fake, None, None, None, 7, fake, need, None) == 1
    assert lib.moe_w4a8_gemm1_partials(fake, fake, ctypes.byref(d), fake, fake, 3, fake, 3, fake, need, None) == 1
    assert lib.moe_w4a8_gemm2_partials(fake, fake, ctypes.byref(d), fake, 3, fake, -2, fake, need, None) == 1
    # the status query needs an aligned workspace of at least the header; NULL names the no-alloc
    # array, whose address lookup needs a device (MOE_ERR_CUDA without one, nothing dereferenced)
    import torch
    assert lib.moe_w4a8_device_status(None, 0, None) == (0 if torch.cuda.is_available() else 4)
    assert lib.moe_w4a8_device_status(ctypes.c_void_p(0x100010), 1024, None) == 1
    assert lib.moe_w4a8_device_status(fake, 16, None) == 1


def test_host_buffer_entry_checks_before_touching_memory(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(4, 2048, 512, 512, 1, 10, 128)
    need = lib.moe_w4a8_workspace_size(ctypes.byref(d))
    need_host = lib.moe_w4a8_forward_host_workspace_size(ctypes.byref(d))
    # the staged inputs (T*H int8, T floats, T*E floats) and output (T*H floats) on top, 256-aligned
    assert need_host % 256 == 0
    assert need_host >= need + d.T * d.H + 4 * d.T + 4 * d.T * d.E + 4 * d.T * d.H
    d_bad = binding.dims_of(4, 2048, 512, 512, 1, 10, 48)
    assert lib.moe_w4a8_forward_host_workspace_size(ctypes.byref(d_bad)) == 0
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: the checks fail first
    odd = ctypes.c_void_p(0x100008)
    args = [fake] * 7
    assert lib.moe_w4a8_forward_host(odd, *args[1:], ctypes.byref(d), fake, fake, need_host, None) == 1
    assert lib.moe_w4a8_forward_host(*args, ctypes.byref(d), None, fake, need_host, None) == 1
    assert lib.moe_w4a8_forward_host(*args, ctypes.byref(d), fake, ctypes.c_void_p(0x100010), need_host, None) == 1
    # the plain layer workspace is not enough: the staging area comes on top
    assert lib.moe_w4a8_forward_host(*args, ctypes.byref(d), fake, fake, need, None) == 3
    d0 = binding.dims_of(0, 2048, 512, 512, 1, 10, 128)
    assert lib.moe_w4a8_forward_host(None, None, None, fake, fake, fake, fake, ctypes.byref(d0), None, None, 0, None) == 0


def test_bf16_entry_checks_its_arguments(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(4, 2048, 512, 512, 1, 10, 128)
    need = lib.moe_w4a8_workspace_size(ctypes.byref(d))
    need_bf16 = lib.moe_w4a8_forward_bf16_workspace_size(ctypes.byref(d))
    assert need_bf16 % 256 == 0 and need_bf16 >= need + d.T * d.H + 4 * d.T
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: the checks fail first
    w = [fake] * 4
    assert lib.moe_w4a8_forward_bf16(None, fake, *w, ctypes.byref(d), fake, fake, need_bf16, None) == 1
    assert lib.moe_w4a8_forward_bf16(ctypes.c_void_p(0x100008), fake, *w, ctypes.byref(d), fake, fake, need_bf16,
                                     None) == 1
    assert lib.moe_w4a8_forward_bf16(fake, fake, *w, ctypes.byref(d), fake, fake, need, None) == 3
    d0 = binding.dims_of(0, 2048, 512, 512, 1, 10, 128)
    assert lib.moe_w4a8_forward_bf16(None, None, *w, ctypes.byref(d0), None, None, 0, None) == 0


def test_mixed_bank_entry_checks_its_arguments(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(4, 2048, 512, 512, 1, 10, 128)
    need = lib.moe_w4a8_workspace_size(ctypes.byref(d))
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: the checks fail first
    args = [fake] * 7
    assert lib.moe_w4a8_forward_w2w4(*args, None, ctypes.byref(d), fake, fake, need, None) == 1
    assert lib.moe_w4a8_forward_w2w4(*args, fake, ctypes.byref(d), fake, fake, need - 256, None) == 3
    # sizes neither the decode engine (T <= 32) nor the tcgen05 engine (g a multiple of 128) takes are
    # refused before anything is enqueued
    big = binding.dims_of(4096, 2048, 512, 512, 1, 10, 64)
    need_big = lib.moe_w4a8_workspace_size(ctypes.byref(big))
    assert lib.moe_w4a8_forward_w2w4(*args, fake, ctypes.byref(big), fake, fake, need_big, None) == 2


def test_compact_mixed_bank_layout_matches_the_generators_compaction(lib):
    """The host layout helper (no device work): the same per-slot offsets and bank sizes as the seeded
    generator's own compaction of a mixed bank, and its argument checks."""
    import numpy as np
    import torch
    from bit_moe_expert_router_gb300 import binding, synth
    w = synth.Workload("layout_mixed", T=1, H=256, I=128, E=6, S=1, top_k=2, group=64, twobit_frac=0.5)
    bank = synth.make_bank(w, pack2=True)
    assert 0 < (bank.slot_bits == 2).sum() < w.E
    w13c, o13, w2c, o2 = synth.compact_bank(bank)
    d = binding.dims_of(w.T, w.H, w.I, w.E, w.S, w.top_k, w.group)
    g13, g2, n13, n2 = binding.moe_w4a8_mixed_bank_layout(torch.from_numpy(bank.slot_bits.copy()), d)
    assert np.array_equal(g13.numpy(), o13) and np.array_equal(g2.numpy(), o2)
    assert (n13, n2) == (w13c.size, w2c.size)
    assert np.all(g13.numpy() % 16 == 0) and np.all(g2.numpy() % 16 == 0)
    # each offset a multiple of its slot's row length (the tcgen05 engine's tiles address a slot's rows
    # from offset / row length)
    rl13 = np.where(bank.slot_bits == 2, w.H // 4, w.H // 2)
    rl2 = np.where(bank.slot_bits == 2, w.I // 4, w.I // 2)
    assert np.all(g13.numpy() % rl13 == 0) and np.all(g2.numpy() % rl2 == 0)
    # a 2-bit slot takes half the bytes of a 4-bit one in both banks
    n4 = int((bank.slot_bits == 4).sum())
    assert n13 == (2 * n4 + (w.E + w.S - n4)) * 2 * w.I * w.H // 4
    # the compacted rows are the uniform rows cut to the slot's width
    e2 = int(np.nonzero(bank.slot_bits == 2)[0][0])
    row = w13c[o13[e2] + 3 * (w.H // 4): o13[e2] + 4 * (w.H // 4)]
    assert np.array_equal(row, bank.w13[e2, 3, : w.H // 4])
    bits = np.ascontiguousarray(bank.slot_bits)
    i64 = ctypes.c_int64()
    o = np.empty(w.E + w.S, np.int64)
    assert lib.moe_w4a8_mixed_bank_layout(None, ctypes.byref(d), o.ctypes.data, o.ctypes.data, ctypes.byref(i64),
                                          ctypes.byref(i64)) == 1
    bad = binding.dims_of(1, 256, 96, 6, 1, 2, 32)  # I not a multiple of 64
    assert lib.moe_w4a8_mixed_bank_layout(bits.ctypes.data, ctypes.byref(bad), o.ctypes.data, o.ctypes.data,
                                          ctypes.byref(i64), ctypes.byref(i64)) == 2


def test_compact_mixed_bank_entry_checks_its_arguments(lib):
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(4, 2048, 512, 512, 1, 10, 128)
    need = lib.moe_w4a8_workspace_size(ctypes.byref(d))
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: the checks fail first
    x = [fake] * 3
    # null offsets or slot widths: invalid before anything is enqueued
    assert lib.moe_w4a8_forward_w2w4_compact(*x, fake, None, fake, fake, fake, fake, fake, ctypes.byref(d), fake,
                                             fake, need, None) == 1
    assert lib.moe_w4a8_forward_w2w4_compact(*x, fake, fake, fake, fake, None, fake, fake, ctypes.byref(d), fake,
                                             fake, need, None) == 1
    assert lib.moe_w4a8_forward_w2w4_compact(*x, fake, fake, fake, fake, fake, fake, None, ctypes.byref(d), fake,
                                             fake, need, None) == 1
    assert lib.moe_w4a8_forward_w2w4_compact(*x, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(d), fake,
                                             fake, need - 256, None) == 3
    big = binding.dims_of(4096, 2048, 512, 512, 1, 10, 64)
    need_big = lib.moe_w4a8_workspace_size(ctypes.byref(big))
    assert lib.moe_w4a8_forward_w2w4_compact(*x, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(big), fake,
                                             fake, need_big, None) == 2


def test_plain_c_program_links_against_the_library(cuda_lib, tmp_path):
    """The boundary is a C ABI: a C11 program includes the header, links the library and calls it
    (host-side entry points only: no GPU is needed for these)."""
    import shutil
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi_check.c"
    src.write_text(r'''
#include <stdio.h>
#include "moe_w4a8.h"
int main(void) {
    moe_dims_t d = {4, 2048, 512, 512, 1, 10, 128};
    moe_dims_t bad = {4, 2048, 512, 512, 1, 10, 48};
    if (moe_w4a8_version() != MOE_W4A8_ABI_VERSION) return 1;
    if (moe_w4a8_workspace_size(&d) == 0 || moe_w4a8_workspace_size(&bad) != 0) return 2;
    if (moe_w4a8_forward_host_workspace_size(&d) <= moe_w4a8_workspace_size(&d)) return 3;
    /* host-detected errors come back before anything is enqueued */
    if (moe_w4a8_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, &d, NULL, NULL, 0, NULL) != MOE_ERR_INVALID_ARG)
        return 4;
    printf("%s|%s\n", moe_w4a8_status_string(MOE_OK), moe_w4a8_status_string(MOE_ERR_WORKSPACE_TOO_SMALL));
    return 0;
}
''')
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(cuda_lib)
    libname = os.path.basename(cuda_lib)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", str(src), "-I", os.path.join(REPO, "include"),
                    "-o", str(exe), os.path.join(libdir, libname), f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == "ok|workspace too small"


def test_binding_checks_tensors_before_calling_the_library(lib):
    """The Python binding refuses wrong dtypes, shapes, devices and layouts itself (no CUDA call)."""
    import torch
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(4, 256, 128, 8, 1, 2, 64)
    slots = d.E + d.n_shared
    good = dict(x_q=torch.zeros(4, 256, dtype=torch.int8), x_scale=torch.zeros(4), logits=torch.zeros(4, 8),
                w13=torch.zeros(slots, 256, 128, dtype=torch.uint8), s13=torch.zeros(slots, 256, 4),
                w2=torch.zeros(slots, 256, 64, dtype=torch.uint8), s2=torch.zeros(slots, 256, 2),
                out=torch.zeros(4, 256))
    ws = torch.zeros(1024, dtype=torch.uint8)

    def call(**over):
        a = dict(good, **over)
        return binding.moe_w4a8_forward(a["x_q"], a["x_scale"], a["logits"], a["w13"], a["s13"], a["w2"], a["s2"],
                                        d, a["out"], ws)

    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        call()                                                   # host tensors go through moe_w4a8_forward_host
    with pytest.raises(TypeError, match="x_q: dtype"):
        call(x_q=torch.zeros(4, 256))
    with pytest.raises(ValueError, match="x_q is required"):
        call(x_q=None)
    # the host-buffer entry wants CPU activations and checks their shapes and layouts the same way
    with pytest.raises(ValueError, match="router_logits must be a contiguous CPU tensor"):
        binding.moe_w4a8_forward_host(good["x_q"], good["x_scale"], torch.zeros(8, 4).t(), good["w13"], good["s13"],
                                      good["w2"], good["s2"], d, good["out"], ws)
    with pytest.raises(ValueError, match="out must be a contiguous CPU tensor"):
        binding.moe_w4a8_forward_host(good["x_q"], good["x_scale"], good["logits"], good["w13"], good["s13"],
                                      good["w2"], good["s2"], d, torch.zeros(4, 255), ws)


def test_binding_checks_the_compact_bank_entry(lib):
    """The compact mixed-bank entry refuses wrong arguments in the binding itself (no CUDA call: on a
    machine without a GPU the first argument's checks are the ones reached), and the layout helper
    wants the slot widths as a host tensor of E+S entries."""
    import torch
    from bit_moe_expert_router_gb300 import binding
    d = binding.dims_of(4, 256, 128, 8, 1, 2, 64)
    slots = d.E + d.n_shared
    args = [torch.zeros(4, 256, dtype=torch.int8), torch.zeros(4), torch.zeros(4, 8),
            torch.zeros(4096, dtype=torch.uint8), torch.zeros(slots, dtype=torch.int64), torch.zeros(slots, 256, 4),
            torch.zeros(4096, dtype=torch.uint8), torch.zeros(slots, dtype=torch.int64), torch.zeros(slots, 256, 2),
            torch.full((slots,), 4, dtype=torch.uint8)]
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError, match="x_q must be a CUDA tensor"):
        binding.moe_w4a8_forward_w2w4_compact(*args, d, torch.zeros(4, 256), ws)
    with pytest.raises(TypeError, match="x_q: dtype"):
        binding.moe_w4a8_forward_w2w4_compact(torch.zeros(4, 256), *args[1:], d, torch.zeros(4, 256), ws)
    with pytest.raises(ValueError, match="slot_bits must be a contiguous CPU tensor"):
        binding.moe_w4a8_mixed_bank_layout(torch.full((slots - 1,), 4, dtype=torch.uint8), d)
    with pytest.raises(TypeError, match="slot_bits: dtype"):
        binding.moe_w4a8_mixed_bank_layout(torch.full((slots,), 4, dtype=torch.int32), d)


def test_binding_checks_the_workspace_and_the_device(lib):
    """Every call needs a CUDA uint8 workspace and all device tensors on one device (checked before any call)."""
    import torch
    from bit_moe_expert_router_gb300 import binding
    with pytest.raises(ValueError, match="workspace must be a CUDA tensor"):
        binding._ws_view(torch.zeros(1024, dtype=torch.uint8))
    with pytest.raises(TypeError, match="workspace: dtype"):
        binding._ws_view(torch.zeros(1024))
    a, b = torch.zeros(4), torch.zeros(4, device="meta")
    assert binding._one_device("f", (a, None, a)) == a.device
    with pytest.raises(ValueError, match="share one device"):
        binding._one_device("moe_w4a8_forward", (a, None, b))


def test_binding_calls_on_the_tensors_device_with_its_stream(monkeypatch):
    """_call appends the current stream of the tensors' device, makes that device current only when it is
    not, and turns a non-zero status into MoeError (fakes stand in for the library and the CUDA runtime)."""
    import contextlib
    import types
    import torch
    from bit_moe_expert_router_gb300 import binding
    calls, switched = [], []

    class FakeLib:
        def moe_w4a8_forward(self, *args):
            calls.append(args)
            return self.status

        def moe_w4a8_status_string(self, status):
            return b"fake status"

    lib = FakeLib()
    monkeypatch.setattr(binding, "_load", lambda: lib)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda dev: types.SimpleNamespace(cuda_stream=100 + dev.index))

    @contextlib.contextmanager
    def fake_device(dev):
        switched.append(dev.index)
        yield

    monkeypatch.setattr(torch.cuda, "device", fake_device)
    on = lambda i: types.SimpleNamespace(device=torch.device("cuda", i))  # noqa: E731

    lib.status = 0
    binding._call("moe_w4a8_forward", (on(0), None, on(0)), "a", "b")
    assert calls[-1][:2] == ("a", "b") and calls[-1][2].value == 100 and switched == []
    binding._call("moe_w4a8_forward", (on(1), on(1)), "c")
    assert calls[-1][0] == "c" and calls[-1][1].value == 101 and switched == [1]
    lib.status = 3
    with pytest.raises(binding.MoeError):
        binding._call("moe_w4a8_forward", (on(0),), "d")
    n = len(calls)
    with pytest.raises(ValueError, match="share one device"):
        binding._call("moe_w4a8_forward", (on(0), on(1)), "e")
    assert len(calls) == n                       # refused before the library is called


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No CPU fallback: with the CUDA library absent every entry point raises before doing anything."""
    import torch
    from bit_moe_expert_router_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libmoe_w4a8.so"))
    d = binding.dims_of(4, 256, 128, 8, 0, 2, 64)
    with pytest.raises(RuntimeError, match="is missing"):
        binding.moe_w4a8_version()
    with pytest.raises(RuntimeError, match="is missing"):
        binding.moe_w4a8_workspace_size(d)
    with pytest.raises(RuntimeError, match="is missing"):
        binding.Layer(d, None, None, None, None, "cpu")


def test_engine_query_without_a_device_returns_cleanly(lib):
    """Host-only: with no usable device the engine query still answers (the decode engine needs the
    device's shared-memory size, so it is ruled out) and invalid sizes give -1."""
    import torch
    from bit_moe_expert_router_gb300 import binding
    if torch.cuda.is_available():
        pytest.skip("a device is visible")
    d = binding.dims_of(4, 2048, 512, 512, 1, 10, 128)
    assert binding.moe_w4a8_engine_for(d) in (binding.ENGINE_TCGEN05, binding.ENGINE_GROUPED)
    d.group = 48
    assert binding.moe_w4a8_engine_for(d) == -1


def test_binding_refuses_a_library_of_another_abi_version(monkeypatch, lib):
    """The binding and the library move in lock-step: a different ABI version is refused at load."""
    from bit_moe_expert_router_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "ABI_VERSION", lib.moe_w4a8_version() + 1)
    with pytest.raises(RuntimeError, match="ABI version"):
        binding._load()
