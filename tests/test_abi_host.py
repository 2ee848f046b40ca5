"""Host-side tests of the C-ABI library (no GPU): symbol exports, the C++
planner bit-exact against the oracle's staging, and argument/limit errors."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import staging as S
from prefill_only_shared_gb300.workloads import make_workload

from conftest import ROOT
from test_oracle_staging import csr, golden_staging, random_case

HEADER = os.path.join(ROOT, "include", "sp.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sp_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    L = ctypes.CDLL(lib.lib()._name)
    syms = declared_symbols()
    assert len(syms) >= 15
    for s in syms:
        assert hasattr(L, s), f"libsp.so does not export {s}"
    # and the binding declares a signature for each
    assert set(syms) == set(lib.SIGNATURES)


def test_status_strings(lib):
    for code in range(8):
        assert lib.sp_status_str(code) and lib.sp_status_str(code) != "unknown status"


SHAPE = dict(n_q_heads=8, n_kv_heads=2, head_dim=64, page_size=16, hidden=512, vocab=4096)


def build_both(lib, req, off, toks, shape=SHAPE, max_pages=1 << 20):
    plan = lib.sp_plan_build(lib.make_shape(**shape), req, off, toks, max_pages)
    ref = S.build_plan(req, off, toks)
    return plan, ref


def assert_plan_equal(plan, ref):
    assert plan.rounds() == ref.rounds
    seg = plan.segments()
    assert len(seg["len"]) == len(ref.segments)
    for i, s in enumerate(ref.segments):
        assert seg["node_start"][i] == s.node_start
        assert seg["len"][i] == s.length
        assert seg["parent"][i] == s.parent
        assert seg["shared"][i] == int(s.shared)
        assert seg["req"][i] == s.req
        expect_round = ref.claimed_round[i] if s.shared else ref.branch_round[s.members[0]]
        assert seg["round"][i] == expect_round
    br = plan.branches()
    for b in range(len(ref.paths)):
        assert br["last_seg"][b] == ref.paths[b][-1]
        assert br["last_row"][b] == ref.branch_last_row(b)
        assert br["round"][b] == ref.branch_round[b]
        assert br["recompute"][b] == int(ref.recompute[b])
    st = plan.stats()
    rs = S.plan_stats(ref)
    for k in ("logical_tokens", "computed_tokens", "reused_tokens", "node_tokens", "n_segments",
              "n_shared_segments", "n_rounds"):
        assert st[k] == rs[k], k


def test_planner_printed_example(lib):
    g, seqs = golden_staging()
    off, toks = csr(seqs)
    plan, ref = build_both(lib, np.zeros(len(seqs), np.int32), off, toks)
    assert_plan_equal(plan, ref)
    names = g["branch_names"]
    assert [[names[b] for b in r] for r in plan.rounds()] == g["printed_rounds"]


@pytest.mark.parametrize("seed", range(80))
def test_planner_random_tries_bit_exact(lib, seed):
    req, seqs = random_case(seed)
    off, toks = csr(seqs)
    plan, ref = build_both(lib, req, off, toks)
    assert_plan_equal(plan, ref)


@pytest.mark.parametrize("name", ["tiny", "yesno", "choice64", "tree2", "batch64"])
def test_planner_configs_bit_exact(lib, name):
    wl = make_workload(name, tokens_only=True)
    sh = wl.shape
    shape = dict(n_q_heads=sh.n_q_heads, n_kv_heads=sh.n_kv_heads, head_dim=sh.head_dim,
                 page_size=sh.page_size, hidden=sh.hidden, vocab=sh.vocab)
    plan, ref = build_both(lib, wl.req_of_branch, wl.tok_offsets, wl.tokens, shape)
    assert_plan_equal(plan, ref)
    seg = plan.segments()
    # every segment starts on a fresh page, pages consecutive
    pages = np.ceil(seg["len"] / 16).astype(np.int64)
    assert (seg["first_page"] == np.concatenate([[0], np.cumsum(pages)[:-1]])).all()
    assert plan.stats()["pages_used"] == int(pages.sum())


def test_planner_errors(lib):
    sh = lib.make_shape(**SHAPE)
    off, toks = csr([[1, 2, 3], [1, 2, 4]])
    req = np.zeros(2, np.int32)
    # pool too small
    with pytest.raises(lib.SpError) as e:
        lib.sp_plan_build(sh, req, off, toks, max_pages=2)
    assert e.value.status == 3
    assert lib.sp_plan_build(sh, req, off, toks, max_pages=3).stats()["pages_used"] == 3
    # bad shapes
    for bad in (dict(SHAPE, head_dim=96), dict(SHAPE, n_q_heads=6, n_kv_heads=4),
                dict(SHAPE, page_size=32), dict(SHAPE, hidden=100)):
        with pytest.raises(lib.SpError) as e:
            lib.sp_plan_build(lib.make_shape(**bad), req, off, toks, 100)
        assert e.value.status == 1
    # empty branch
    off2, toks2 = csr([[1, 2], []])
    with pytest.raises(lib.SpError) as e:
        lib.sp_plan_build(sh, req, off2, toks2, 100)
    assert e.value.status == 1
    # per-branch limit 32768 tokens, per-request limit 262144 tokens
    off3, toks3 = csr([np.arange(32769) % 7])
    with pytest.raises(lib.SpError) as e:
        lib.sp_plan_build(sh, np.zeros(1, np.int32), off3, toks3, 1 << 20)
    assert e.value.status == 2
    seqs = [np.full(32768, i, np.int32) for i in range(9)]
    off4, toks4 = csr(seqs)
    with pytest.raises(lib.SpError) as e:
        lib.sp_plan_build(sh, np.zeros(9, np.int32), off4, toks4, 1 << 20)
    assert e.value.status == 2
    # same branches split over two requests are within limits
    assert lib.sp_plan_build(sh, np.array([0] * 5 + [1] * 4, np.int32), off4, toks4,
                             1 << 20).stats()["n_requests"] == 2


def test_check_labels(lib):
    lib.sp_check_labels([0, 2, 5], [1, 2, 3, 4, 4], 10)
    for off, ids in (([0, 1, 3], [1, 2, 3]), ([0, 2, 4], [1, 2, 3, 10]), ([0, 2, 4], [1, -1, 3, 4]),
                     ([0, 65], list(range(65)))):
        with pytest.raises(lib.SpError):
            lib.sp_check_labels(off, ids, 10 if len(ids) < 65 else 100)


def test_split_plan_covers_all_units(lib):
    """The planner's tiles (after splitting) cover each tile's KV units exactly
    once; checked through the descriptor image semantics on the host."""
    wl = make_workload("yesno", tokens_only=True)
    sh = wl.shape
    plan = lib.sp_plan_build(lib.make_shape(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, 16,
                                            sh.hidden, sh.vocab), wl.req_of_branch,
                             wl.tok_offsets, wl.tokens, 1 << 20, n_sms=152)
    st = plan.stats()
    assert st["attn_workspace_bytes"] > 0 and st["desc_bytes"] > 0


def test_check_options(lib):
    """Host validation of the option CSRs of sp_option_softmax."""
    lib.sp_check_options([0, 1, 3, 4, 6], 6, [0, 2, 4])
    for opt_off, n_rows, q_off in (([1, 2, 3], 3, [0, 2]),        # opt_off must start at 0
                                   ([0, 1, 1, 2], 2, [0, 3]),     # an empty option
                                   ([0, 1, 2], 1, [0, 2]),        # rows past n_rows
                                   ([0, 1, 2, 3], 3, [0, 1, 3]),  # a question of 1 option
                                   ([0, 1, 2], 2, [0, 3]),        # options past n_opts
                                   ([0] + list(range(1, 67)), 66, [0, 66])):  # 66 options
        with pytest.raises(lib.SpError):
            lib.sp_check_options(opt_off, n_rows, q_off)


def test_struct_layouts_match_the_header(lib, tmp_path):
    """The ctypes structures of the binding have the C compiler's size and
    field offsets for every struct the header declares by value."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"sp_shape": lib.sp_shape, "sp_plan_stats": lib.sp_plan_stats,
               "sp_input_set": lib.sp_input_set}
    lines = ["#include <stdio.h>", "#include <stddef.h>", f'#include "{HEADER}"',
             "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{name}.{f} %zu\\n", offsetof({name}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-o", str(exe), str(src)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                  text=True).stdout.splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
        for f, _ in cls._fields_:
            assert int(got[f"{name}.{f}"]) == getattr(cls, f).offset, (name, f)


def test_host_pass_checks_before_any_copy(lib):
    """sp_run_pass_host validates the host label CSR and every capacity (the
    input set's included) before it enqueues anything: these calls return
    before any CUDA call, so the device pointers are placeholders that are
    never dereferenced."""
    sh = lib.make_shape(8, 2, 64, 16, 64, 100)
    off, toks = csr([[1, 2, 3, 4], [1, 2, 3, 5]])
    req = np.zeros(2, np.int32)
    T = 5  # node rows: 3 shared + 1 + 1
    q = np.zeros(T * 8 * 64, np.uint16)
    k = np.zeros(T * 2 * 64, np.uint16)
    h = np.zeros(2 * 64, np.uint16)
    lab_off = np.array([0, 2, 4], np.int32)
    lab_ids = np.array([1, 2, 3, 4], np.int32)
    probs_h = np.zeros(4, np.float32)
    am_h = np.zeros(2, np.int32)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced on these paths

    def call(lab_off, lab_ids, q_rows, desc_host_bytes=1 << 20):
        iset = lib.sp_input_set(q=fake, k=fake, v=fake, h=fake, label_off=fake, label_ids=fake,
                                q_rows=q_rows, h_rows=2, labels_cap=4, desc_host=fake,
                                desc_host_bytes=desc_host_bytes, done_event=fake,
                                copied_event=fake)
        st = lib.sp_plan_stats()
        P = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        status = lib.lib().sp_run_pass_host(
            ctypes.byref(sh), 2, req.ctypes.data_as(lib._I32P), off.ctypes.data_as(lib._I64P),
            toks.ctypes.data_as(lib._I32P), T, P(q), P(k), P(k), P(h),
            lab_off.ctypes.data_as(ctypes.c_void_p), lab_ids.ctypes.data_as(ctypes.c_void_p),
            len(lab_ids), ctypes.byref(iset), fake, 1 << 20, fake, fake, fake, 1 << 20, fake,
            1 << 24, fake, fake, fake, fake, 1 << 26, fake, fake, P(probs_h), P(am_h), None, None,
            ctypes.byref(st))
        return status, st.as_dict()

    # a label count of 1, an id past the vocabulary, offsets that do not end at n_labels
    for lo, li in (([0, 1, 4], [1, 2, 3, 4]), ([0, 2, 4], [1, 2, 3, 100]),
                   ([0, 2, 3], [1, 2, 3, 4])):
        assert call(np.array(lo, np.int32), np.array(li, np.int32), T)[0] == 1
    # the input set holds fewer node rows than the pass: SP_ERR_WORKSPACE, stats filled
    status, st = call(lab_off, lab_ids, T - 1)
    assert status == 7 and st["node_tokens"] == T and st["n_branches"] == 2
    # descriptor staging shorter than the plan's descriptor
    status, st = call(lab_off, lab_ids, T, desc_host_bytes=st["desc_bytes"] - 1)
    assert status == 7


def test_run_pass_checks_before_any_launch(lib):
    """sp_run_pass reports a node-row count that differs from the plan's
    (SP_ERR_ARG), a pool smaller than the plan (SP_ERR_POOL_FULL, with the
    pages needed in the stats) and short descriptor / workspace buffers
    (SP_ERR_WORKSPACE, with the sizes needed) before anything is enqueued; the
    device pointers are placeholders that these paths never dereference."""
    sh = lib.make_shape(8, 2, 64, 16, 64, 100)
    off, toks = csr([[1, 2, 3, 4], [1, 2, 3, 5]])
    req = np.zeros(2, np.int32)
    fake = ctypes.c_void_p(1 << 20)

    def call(node_rows, pool_pages=1 << 20, desc_bytes=1 << 20, attn_ws=1 << 24, lm_ws=1 << 26,
             h=fake):
        st = lib.sp_plan_stats()
        status = lib.lib().sp_run_pass(
            ctypes.byref(sh), 2, req.ctypes.data_as(lib._I32P), off.ctypes.data_as(lib._I64P),
            toks.ctypes.data_as(lib._I32P), node_rows, fake, fake, fake, fake, pool_pages, fake,
            fake, fake, desc_bytes, fake, attn_ws, h, fake, fake, fake, 4, fake, fake, fake,
            lm_ws, fake, fake, None, ctypes.byref(st))
        return status, st.as_dict()

    # the readout's own checks come before the plan too: h not 16-byte aligned
    status, st = call(5, h=ctypes.c_void_p((1 << 20) + 8))
    assert status == 1 and st["node_tokens"] == 0

    status, st = call(4)
    assert status == 1 and st["node_tokens"] == 5
    status, st = call(5, pool_pages=2)
    assert status == 3 and st["pages_used"] == 3
    status, st = call(5, desc_bytes=16)
    assert status == 7 and st["desc_bytes"] > 16
    assert call(5, lm_ws=0)[0] == 7


def test_plain_c_caller(lib, tmp_path):
    """tests/c_abi_host.c, a C99 program that includes only sp.h and links
    only libsp, plans two requests, checks their rounds and token accounting,
    runs the batcher and checks the error codes (host-only entry points)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lib.lib()._name)
    exe = tmp_path / "c_abi_host"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_host.c"), "-L", libdir, "-lsp",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "passed" in r.stdout
