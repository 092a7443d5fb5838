"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/cpattn.h declares, and rejects invalid arguments
synchronously, before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def cp():
    import __graft_entry__
    __graft_entry__.build()
    import blockwise_online_softmax_cpattn_gb300 as mod
    return mod


def _declared_functions():
    with open(os.path.join(ROOT, "include", "cpattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpattn_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(cp):
    names = _declared_functions()
    assert len(names) >= 13
    lib = ctypes.CDLL(cp.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def _desc(mod, **kw):
    base = dict(B=1, H_q=4, H_kv=2, T=512, D=64, cp=2, layout="zigzag", dtype="bf16")
    base.update(kw)
    return mod.make_desc(**base)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("kw,code", [
    (dict(H_q=3, H_kv=2), 1),
    (dict(T=502), 1),                        # zigzag needs T % (2 cp) == 0
    (dict(T=511, layout="contiguous"), 1),   # T % cp != 0
    (dict(D=192), 2),
    (dict(causal=0), 2),
    (dict(scale=0.0), 1),
    (dict(scale=-1.0), 1),
    (dict(cp=0), 1),
    (dict(a2a=3, cp=2), 1),                  # a2a must divide cp
    (dict(a2a=2, cp=4, H_kv=1, H_q=4), 1),   # heads must split over a2a
    (dict(a2a=4, cp=4, H_kv=2, H_q=8), 1),   # full Ulysses (a2a = cp): H_kv % cp != 0
    (dict(layout=7), 1),
    (dict(dtype=5), 1),
    (dict(B=0), 1),
])
def test_invalid_descriptors_are_rejected(cp, kw, code):
    d = _desc(cp, **kw)
    assert cp.cpattn_ring_fwd(d, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == code
    assert cp.cpattn_ring_bwd(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              1 << 30, 0) == code
    assert cp.cpattn_partial_fwd(d, 0, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == code
    assert cp.cpattn_ring_bwd_workspace(d) == 0
    assert cp.cpattn_allgather_fwd(d, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == code
    assert cp.cpattn_allgather_bwd(d, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0,
                                   FAKE, 1 << 30, 0) == code
    assert cp.cpattn_allgather_bwd_workspace(d) == 0


def test_null_and_misaligned_pointers(cp):
    d = _desc(cp)
    assert cp.cpattn_ring_fwd(d, 0, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert cp.cpattn_ring_fwd(d, FAKE + 8, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert cp.cpattn_merge(10, 64, FAKE, FAKE, FAKE + 4, FAKE, FAKE, FAKE, 0) == 1
    assert cp.cpattn_merge(-1, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert cp.cpattn_merge(0, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 0  # nothing to do
    assert cp.cpattn_layout(0, d, FAKE, FAKE, 4, 0) == 1                    # src == dst
    assert cp.cpattn_layout(9, d, FAKE, FAKE + 64, 4, 0) == 1
    assert cp.cpattn_layout(2, _desc(cp, a2a=2, cp=4, T=512), FAKE, FAKE + 64, 3, 0) == 1


def test_ranks_and_workspace_are_checked(cp):
    d = _desc(cp)
    assert cp.cpattn_partial_fwd(d, 2, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert cp.cpattn_partial_fwd(d, 0, -1, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    need = cp.cpattn_ring_bwd_workspace(d)
    assert need >= 1 * 4 * 512 * 4 and need % 256 == 0
    assert cp.cpattn_ring_bwd(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              need - 1, 0) == 1


def test_status_strings(cp):
    for code in range(5):
        assert cp.cpattn_status_string(code)
    assert cp.cpattn_status_string(99) == "unknown status"


def test_timing_table_host_side(cp):
    assert cp.cpattn_timing_reset() == 0
    assert cp.cpattn_timing_enable(False) == 0
    assert cp.cpattn_timing_collect() == 0
    assert cp.cpattn_timing_table() == {}


def test_allgather_ranks_flags_and_workspace_are_checked(cp):
    d = _desc(cp)  # cp = 2: ranks 0 and 1
    assert cp.cpattn_allgather_fwd(d, 2, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert cp.cpattn_allgather_fwd(d, -1, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert cp.cpattn_allgather_fwd(d, 0, FAKE, FAKE, FAKE, FAKE + 8, FAKE, 0) == 1
    need = cp.cpattn_allgather_bwd_workspace(d)
    # Delta and the base-2 LSE of one rank's rows: B * H_q * T / cp floats each
    assert need >= 2 * 1 * 4 * 256 * 4 and need % 256 == 0
    assert need < cp.cpattn_ring_bwd_workspace(d)
    args = [FAKE] * 8
    assert cp.cpattn_allgather_bwd(d, 2, *args, 0, FAKE, need, 0) == 1
    assert cp.cpattn_allgather_bwd(d, 0, *args, 2, FAKE, need, 0) == 1      # accumulate: 0 or 1
    assert cp.cpattn_allgather_bwd(d, 0, *args, 1, FAKE, need - 1, 0) == 1  # workspace too small
    assert cp.cpattn_allgather_bwd(d, 0, *args[:7], 0, 1, FAKE, need, 0) == 1  # null dv_sum


def test_packed_arguments_are_checked(cp):
    d = _desc(cp)
    need = cp.cpattn_packed_workspace(d)
    # documents of every position (lo, hi: int32 each), the work orders of the
    # 128-token tiles (int32 each), then the backward statistics
    # (each section rounded up to 256 bytes: B1 T512 gives 2 x 2048 + 2 x 256)
    assert need == 2 * 2048 + 2 * 256 + cp.cpattn_ring_bwd_workspace(d)
    assert cp.cpattn_packed_workspace(_desc(cp, a2a=2, cp=4, T=512)) == 0
    f = [FAKE] * 5
    assert cp.cpattn_ring_fwd_packed(d, FAKE, 0, *f, FAKE, need, 0) == 1      # n_docs < 1
    assert cp.cpattn_ring_fwd_packed(d, 0, 2, *f, FAKE, need, 0) == 1         # null starts
    assert cp.cpattn_ring_fwd_packed(d, FAKE + 2, 2, *f, FAKE, need, 0) == 1  # misaligned starts
    assert cp.cpattn_ring_fwd_packed(d, FAKE, 2, *f, FAKE, need - 1, 0) == 1  # workspace
    assert cp.cpattn_ring_fwd_packed(_desc(cp, a2a=2, cp=4, T=512), FAKE, 2, *f, FAKE, need,
                                     0) == 2
    b = [FAKE] * 9
    assert cp.cpattn_ring_bwd_packed(d, FAKE, 0, *b, FAKE, need, 0) == 1
    assert cp.cpattn_ring_bwd_packed(d, FAKE, 2, *b, FAKE, need - 1, 0) == 1
    assert cp.cpattn_ring_bwd_packed(_desc(cp, causal=0), FAKE, 2, *b, FAKE, need, 0) == 2


def test_layout_batch_arguments_are_checked(cp):
    d = _desc(cp)
    srcs = [FAKE, FAKE + 4096]
    dsts = [FAKE + 8192, FAKE + 12288]
    assert cp.cpattn_layout_batch(0, d, [], [], [], 0) == 1                  # n = 0
    assert cp.cpattn_layout_batch(0, d, [FAKE] * 9, [FAKE + 64] * 9, [4] * 9, 0) == 1  # n > 8
    assert cp.cpattn_layout_batch(0, d, srcs, [dsts[0], srcs[1]], [4, 2], 0) == 1     # src == dst
    assert cp.cpattn_layout_batch(0, d, srcs, dsts, [4, 0], 0) == 1          # no heads
    assert cp.cpattn_layout_batch(0, d, [srcs[0], FAKE + 8], dsts, [4, 2], 0) == 1    # misaligned
    assert cp.cpattn_layout_batch(9, d, srcs, dsts, [4, 2], 0) == 1          # no such permute
    assert cp.cpattn_layout_batch(0, _desc(cp, H_q=3), srcs, dsts, [4, 2], 0) == 1  # descriptor
    lib = ctypes.CDLL(cp.LIB_PATH)
    f = lib.cpattn_layout_batch
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.POINTER(cp.CpattnDesc), ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert f(0, ctypes.byref(d), 1, None, None, None, None) == 1             # null arrays


def test_partial_bwd_arguments_are_checked(cp):
    d = _desc(cp)  # cp = 2
    need = cp.cpattn_partial_bwd_workspace(d)
    assert need == cp.cpattn_allgather_bwd_workspace(d) and need % 256 == 0
    assert cp.cpattn_partial_bwd_stats(d, FAKE, FAKE, FAKE, FAKE, need - 1, 0) == 1
    assert cp.cpattn_partial_bwd_stats(d, FAKE, FAKE + 4, FAKE, FAKE, need, 0) == 1
    assert cp.cpattn_partial_bwd_stats(_desc(cp, D=192), FAKE, FAKE, FAKE, FAKE, need, 0) == 2
    args = [FAKE] * 7
    assert cp.cpattn_partial_bwd(d, 2, 0, *args, 0, FAKE, need, 0) == 1       # q rank
    assert cp.cpattn_partial_bwd(d, 0, -1, *args, 0, FAKE, need, 0) == 1      # kv rank
    assert cp.cpattn_partial_bwd(d, 0, 1, *args, 2, FAKE, need, 0) == 1       # accumulate
    assert cp.cpattn_partial_bwd(d, 0, 1, *args, 1, FAKE, need - 1, 0) == 1   # workspace
    assert cp.cpattn_partial_bwd(d, 0, 1, *args[:6], 0, 0, FAKE, need, 0) == 1  # null dv_part


def test_host_step_arguments_are_checked(cp):
    d = _desc(cp)
    need = cp.cpattn_ring_step_host_workspace(d)
    # staging of q, k, v, dO; layout-order q, k, v, dO, o, LSE, dq, dk, dv; the
    # natural-order LSE; the backward's statistics of one half
    q, k, lse = 1 * 4 * 512 * 64 * 2, 1 * 2 * 512 * 64 * 2, 1 * 4 * 512 * 4
    assert need >= 6 * q + 6 * k + 2 * lse and need % 256 == 0
    assert cp.cpattn_ring_step_host_workspace(_desc(cp, a2a=2, cp=4, T=512)) == 0
    h = [FAKE] * 9
    assert cp.cpattn_ring_step_host(_desc(cp, a2a=2, cp=4, T=512), *h, FAKE, need, 0) == 2
    assert cp.cpattn_ring_step_host(d, *h, FAKE, need - 1, 0) == 1           # workspace size
    assert cp.cpattn_ring_step_host(d, *h, FAKE + 16, need, 0) == 1          # 256-byte alignment
    assert cp.cpattn_ring_step_host(d, *h[:8], 0, FAKE, need, 0) == 1        # null dv
    assert cp.cpattn_ring_step_host(_desc(cp, H_q=3), *h, FAKE, need, 0) == 1


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_compiles_on_its_own(tmp_path, lang, std):
    """include/cpattn.h is a plain C header (no CUDA or torch types in the
    signatures): it compiles alone, warning-free, as C99 and as C++17."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text('#include "cpattn.h"\n'
                   'int main(void) {\n'
                   '  cpattn_status (*f)(void*) = cpattn_check;\n'
                   '  (void)f;\n'
                   '  return 0;\n'
                   '}\n')
    r = subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src),
                        "-o", str(tmp_path / "use.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
