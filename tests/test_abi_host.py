"""The C-ABI library on the host, without a GPU: it loads, exports every
symbol include/zerostep.h declares, its structs match the header, its
partition layout (a host-only function) equals the oracle's independent
layout bit for bit, and invalid arguments are rejected before any device
work is enqueued."""
import ctypes
import os
import random
import re
import subprocess

import pytest

import oracle
from synth.workloads import ALL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zerostep.h")


@pytest.fixture(scope="module")
def zs():
    from zero_partitioned_mixed_step_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_step_gb300 as zs
    zs._abi.lib()
    return zs


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(zero_\w+)\s*\(", text,
                                 re.M)))


def test_exports_every_declared_symbol(zs):
    names = declared_functions()
    assert len(names) == 20, names
    so = ctypes.CDLL(zs._build.LIB)
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(zs._abi.SIGNATURES)


def test_abi_version_matches_header(zs):
    """zero_version() is the version the header states (3: the step state
    carries the scalar cache and is 192 bytes)."""
    m = re.search(r"ABI version: (\d+)", open(HEADER).read())
    assert m and zs._abi.lib().zero_version() == int(m.group(1)) == 3


def test_exports_nothing_else(zs):
    """Only the declared entry points are dynamic symbols of the library
    (it is built with hidden visibility), so internal state such as cached
    launch attributes stays private to each loaded copy."""
    import shutil
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not installed")
    out = subprocess.run([nm, "-D", "--defined-only", zs._build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    exported -= {"_init", "_fini"}
    assert exported == set(declared_functions())


def test_host_alloc_arguments(zs):
    """zero_host_alloc / zero_host_free argument handling that needs no
    device: a zero-byte block is NULL, a NULL result pointer is rejected,
    freeing NULL is a no-op."""
    L = zs._abi.lib()
    p = ctypes.c_void_p(1234)
    assert L.zero_host_alloc(0, ctypes.byref(p)) == 0 and p.value is None
    assert L.zero_host_alloc(64, None) == -1
    assert L.zero_host_free(None) == 0
    assert zs.host_empty(0, zs.torch_dtype(zs.F16)).numel() == 0


def test_bucket_step_validates_before_launch(zs):
    """zero_step_fused_buckets rejects a clipped config, ranges outside the
    layout's buckets and aliased slots before anything is enqueued, and a
    zero-bucket range enqueues nothing."""
    lib = zs._abi.lib()
    E = zs._abi
    lay, _ = zs.zero_partition_layout([100_000, 3], 2, bucket_numel=2 * 8 * 1024)
    assert lay.num_buckets == 7
    fake = 1 << 20
    g2 = (ctypes.c_void_p * 2)(fake, fake)
    slots = (ctypes.c_void_p * 2)(fake, fake + 4096)
    same = (ctypes.c_void_p * 2)(fake, fake)

    def call(first, n, cfg=zs.adam_cfg(), w=slots):
        return lib.zero_step_fused_buckets(g2, 0, 0, ctypes.byref(lay), -1, first, n, w, slots,
                                           slots, slots, ctypes.byref(cfg), fake, None)

    assert call(0, 1, zs.adam_cfg(max_grad_norm=1.0)) == E.EINVAL
    for first, n in ((-1, 1), (0, -1), (7, 1), (6, 2), (0, 8), (1 << 62, 1 << 62)):
        assert call(first, n) == E.EINVAL, (first, n)
    assert call(0, 1, w=same) == E.EINVAL
    assert call(3, 0) == E.OK and call(7, 0) == E.OK


def test_clipped_range_passes_validate_before_launch(zs):
    """The clipped step's range passes reject an unclipped config, ranges
    outside the layout, a second pass with both or neither gradient source,
    misaligned stages and a small workspace before anything is enqueued; a
    zero-bucket range enqueues nothing."""
    lib = zs._abi.lib()
    E = zs._abi
    lay, _ = zs.zero_partition_layout([100_000, 3], 2, bucket_numel=2 * 8 * 1024)
    fake = 1 << 20
    g2 = (ctypes.c_void_p * 2)(fake, fake)
    slots = (ctypes.c_void_p * 2)(fake, fake + 4096)
    clip = zs.adam_cfg(max_grad_norm=1.0)
    wsb = zs.zero_workspace_bytes(lay)

    def p1(first, n, cfg=clip, stage=None, ws_bytes=wsb, grads=g2):
        return lib.zero_step_buckets_pass1(grads, 0, 0, ctypes.byref(lay), -1, first, n, stage,
                                           ctypes.byref(cfg), fake, fake, ws_bytes, None)

    def p2(first, n, cfg=clip, stage=None, grads=g2, ws_bytes=wsb):
        return lib.zero_step_buckets_pass2(grads, 0, 0, ctypes.byref(lay), -1, first, n, slots,
                                           slots, slots, slots, stage, ctypes.byref(cfg), fake,
                                           fake, ws_bytes, None)

    assert p1(0, 1, zs.adam_cfg()) == E.EINVAL and p2(0, 1, zs.adam_cfg()) == E.EINVAL
    for first, n in ((-1, 1), (0, -1), (7, 1), (6, 2)):
        assert p1(first, n) == E.EINVAL and p2(first, n) == E.EINVAL, (first, n)
    assert p1(0, 1, grads=None) == E.EINVAL
    assert p2(0, 1, stage=fake) == E.EINVAL          # both sources
    assert p2(0, 1, grads=None) == E.EINVAL          # neither
    assert p1(0, 1, stage=fake + 16) == E.EALIGN
    assert p2(0, 1, grads=None, stage=fake + 16) == E.EALIGN
    assert p1(0, 1, ws_bytes=wsb - 8) == E.ESPACE and p2(0, 1, ws_bytes=wsb - 8) == E.ESPACE
    assert p1(4, 0) == E.OK and p2(4, 0) == E.OK
    # the norm between the passes: layout, rank and workspace are checked
    assert lib.zero_step_buckets_norm(ctypes.byref(lay), 2, fake, wsb, None) == E.EINVAL
    assert lib.zero_step_buckets_norm(ctypes.byref(lay), -1, fake, wsb - 8, None) == E.ESPACE
    assert lib.zero_step_buckets_norm(ctypes.byref(lay), -1, None, wsb, None) == E.EINVAL


def test_structs_match_header(tmp_path, zs):
    src = tmp_path / "off.c"
    fields = {"zero_layout": zs.Layout, "zero_adam_cfg": zs.AdamCfg,
              "zero_step_state": zs.StepState}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "zerostep.h"', "int main(void){"]
    for cname, cls in fields.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    src.write_text("\n".join(lines))
    exe = tmp_path / "off"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = dict(line.rsplit(" ", 1) for line in subprocess.run(
        [str(exe)], capture_output=True, text=True, check=True).stdout.split("\n") if line)
    for cname, cls in fields.items():
        assert int(out[cname]) == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert int(out[f"{cname}.{f}"]) == getattr(cls, f).offset, (cname, f)


def _same(lay_c, offs_c, lay_o):
    assert lay_c.numel == lay_o.numel
    assert lay_c.flat_numel == lay_o.flat_end
    assert lay_c.padded_numel == lay_o.padded
    assert lay_c.owned_numel == lay_o.owned
    assert lay_c.num_buckets == lay_o.num_buckets
    if lay_o.bucket:
        assert lay_c.slice_numel == lay_o.slice
        assert lay_c.last_slice_numel == lay_o.last_slice
    assert list(offs_c) == list(lay_o.offsets)


@pytest.mark.parametrize("wl", ALL, ids=lambda w: w.name)
def test_layout_matches_oracle_on_workloads(zs, wl):
    lay_c, offs = zs.zero_partition_layout(wl.numels, wl.world, 64, wl.bucket)
    _same(lay_c, offs, oracle.layout(wl.numels, wl.world, 64, wl.bucket))


def test_layout_matches_oracle_random(zs):
    rnd = random.Random(1)
    for _ in range(400):
        world = rnd.choice([1, 2, 3, 4, 7, 8, 16, 64, 100, 1024])
        align = rnd.choice([8, 16, 64, 128])
        numels = [rnd.choice([0, 1, 7, 8, 63, 64, 65, rnd.randint(0, 100000)])
                  for _ in range(rnd.randint(0, 12))]
        bucket = rnd.choice([0, 0, world * 8 * rnd.randint(1, 50)])
        lay_c, offs = zs.zero_partition_layout(numels, world, align, bucket)
        _same(lay_c, offs, oracle.layout(numels, world, align, bucket))


def test_layout_rejects_bad_arguments(zs):
    lib = zs._abi.lib()
    out = zs.Layout()
    arr = (ctypes.c_int64 * 2)(10, 20)
    bad = [(2, arr, 0, 64, 0), (2, arr, 1025, 64, 0), (2, arr, 4, 12, 0), (2, arr, 4, 0, 0),
           (2, arr, 4, 64, 100), (2, arr, 4, 64, -32), (-1, arr, 4, 64, 0), (2, None, 4, 64, 0)]
    for n, a, w, al, b in bad:
        assert lib.zero_partition_layout(n, a, w, al, b, None, ctypes.byref(out)) == zs._abi.EINVAL
    neg = (ctypes.c_int64 * 1)(-5)
    assert lib.zero_partition_layout(1, neg, 4, 64, 0, None, ctypes.byref(out)) == zs._abi.EINVAL


def test_state_init_and_workspace(zs):
    s = zs.zero_state_init(4096.0)
    assert (s.t, s.beta1_pow, s.beta2_pow, s.loss_scale, s.clip_coef, s.cur, s.found_inf) == \
        (0, 1.0, 1.0, 4096.0, 1.0, 0, 0)
    # the library's scalar cache follows the 64 bytes of the state proper, zero-filled
    assert zs.StepState.scalar_cache.offset == 64 and ctypes.sizeof(zs.StepState) == 192
    assert bytes(s)[64:] == bytes(128)
    lib = zs._abi.lib()
    st = zs.StepState()
    for bad in (0.0, -2.0, 3.0, float("inf"), float("nan")):
        assert lib.zero_state_init(ctypes.byref(st), bad) == zs._abi.EINVAL
    assert zs.zero_workspace_bytes() == zs._abi.NOALLOC_SCRATCH_BYTES == 266496
    broken = zs.zero_partition_layout([1000], 2)[0]
    broken.owned_numel += 8
    assert lib.zero_workspace_bytes(ctypes.byref(broken)) == 0
    assert lib.zero_strerror(zs._abi.EALIGN).decode().startswith("buffer")


def _tree_bytes(world, slice_units, last_units, nb):
    """The norm tree's workspace bytes, computed from its definition: chunks
    of at least 512 units (a multiple of 256) sized so a rank has about
    32768 of them, restarting at every bucket slice; 64 chunks per
    superchunk; a 256-byte header, then a double per chunk and per
    superchunk."""
    cd = lambda a, b: -(-a // b)
    units = (nb - 1) * slice_units + last_units
    cu = max(512, cd(cd(units, 32768), 256) * 256)
    cps_last = cd(last_units, cu)
    cps = cd(slice_units, cu) if nb > 1 else cps_last
    cpr = (nb - 1) * cps + cps_last
    spr = cd(cpr, 64)
    return 256 + 8 * world * cpr + 8 * world * spr


@pytest.mark.parametrize("wl", ALL, ids=lambda w: w.name)
def test_workspace_holds_the_norm_tree(zs, wl):
    """zero_workspace_bytes(layout) is the size of the norm's tree for every
    rank of the layout: at most 8 bytes per 4096 elements (2.1 MB for the 8B
    decoder over 8 ranks)."""
    lay, _ = zs.zero_partition_layout(wl.numels, wl.world, 64, wl.bucket)
    if wl.bucket:
        want = _tree_bytes(wl.world, lay.slice_numel // 8, lay.last_slice_numel // 8,
                           lay.num_buckets)
    else:
        want = _tree_bytes(wl.world, lay.owned_numel // 8, lay.owned_numel // 8, 1)
    assert zs.zero_workspace_bytes(lay) == want
    assert want <= lay.padded_numel // 400 + (1 << 16)


def test_entry_points_validate_before_launch(zs):
    """Invalid calls return an error code without touching the device (this
    machine has none, so a launch would fail with a CUDA error instead)."""
    lib = zs._abi.lib()
    lay, _ = zs.zero_partition_layout([1000], 2)
    cfg = zs.adam_cfg()
    fake = 1 << 20  # never dereferenced: validation fails first
    g2 = (ctypes.c_void_p * 2)(fake, fake)
    slots = (ctypes.c_void_p * 2)(fake, fake + 4096)
    same = (ctypes.c_void_p * 2)(fake, fake)
    E = zs._abi
    # rank out of range, dtype, slices without rank
    assert lib.zero_reduce_scatter_sum(g2, 0, 0, ctypes.byref(lay), 2, fake, None) == E.EINVAL
    assert lib.zero_reduce_scatter_sum(g2, 0, 7, ctypes.byref(lay), 0, fake, None) == E.EINVAL
    assert lib.zero_reduce_scatter_sum(g2, 1, 0, ctypes.byref(lay), -1, fake, None) == E.EINVAL
    # misaligned gradient pointer
    g_mis = (ctypes.c_void_p * 2)(fake + 2, fake)
    assert lib.zero_reduce_scatter_sum(g_mis, 0, 0, ctypes.byref(lay), 0, fake, None) == E.EALIGN
    # one-pass step with aliased slots cannot skip bit-exactly
    rc = lib.zero_step_fused(g2, 0, 0, ctypes.byref(lay), -1, same, slots, slots, slots, None,
                             ctypes.byref(cfg), fake, fake, 1 << 20, None)
    assert rc == E.EINVAL
    # workspace too small
    rc = lib.zero_step_fused(g2, 0, 0, ctypes.byref(lay), -1, slots, slots, slots, slots, None,
                             ctypes.byref(cfg), fake, fake, 16, None)
    assert rc == E.ESPACE
    # a staging buffer without clipping
    rc = lib.zero_step_fused(g2, 0, 0, ctypes.byref(lay), -1, slots, slots, slots, slots, fake,
                             ctypes.byref(cfg), fake, fake, 1 << 20, None)
    assert rc == E.EINVAL
    # bad optimizer configuration
    for kw in (dict(beta1=1.0), dict(eps=0.0), dict(lr=-1.0), dict(max_grad_norm=-1.0),
               dict(dynamic_scale=True, backoff=0.3), dict(dynamic_scale=True, growth_interval=0)):
        c = zs.adam_cfg(**kw)
        rc = lib.zero_step_fused(g2, 0, 0, ctypes.byref(lay), -1, slots, slots, slots, slots,
                                 None, ctypes.byref(c), fake, fake, 1 << 20, None)
        assert rc == E.EINVAL, kw
    # a layout whose fields do not agree
    broken = zs.Layout.from_buffer_copy(bytes(lay))
    broken.owned_numel += 8
    assert lib.zero_reduce_scatter_sum(g2, 0, 0, ctypes.byref(broken), -1, fake, None) == E.EINVAL
    assert lib.zero_check_overflow(fake + 4, 10, 1.0, fake, None) == E.EALIGN
    assert lib.zero_grad_norm(fake, 10, 1.0, fake, fake, 8, None) == E.ESPACE
    assert lib.zero_adam_step(fake, fake, fake, fake, fake, 0, -1, ctypes.byref(cfg), fake,
                              None) == E.EINVAL
