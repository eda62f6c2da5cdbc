"""Host-side fault injection (FATHOM_FAULT): a call that would enqueue GPU work
fails after its argument checks with FATHOM_ECUDA and a message naming the
injected fault, and the Python binding raises it as FathomError.  Nothing is
launched, so no GPU is touched; each case runs in a child process because
the library reads the variable once per process."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD_PRELUDE = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, {root!r})
    from bit_plane_kv_gb300 import binding as B
    L = B.lib()
    s = B.make_shape(2, 4096, 128, 4, 512)
    d = ctypes.c_void_p(256)          # never dereferenced: the injected fault comes first
    big = 1 << 40
    def err():
        return L.fathom_last_error().decode()
""")


def run_child(body, fault):
    env = dict(os.environ)
    env.pop("FATHOM_FAULT", None)
    if fault is not None:
        env["FATHOM_FAULT"] = fault
    code = CHILD_PRELUDE.format(root=ROOT) + textwrap.dedent(body)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    return r.stdout


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_plane_kv_gb300 import build as BUILD
    BUILD.build()


def test_every_launching_call_fails_under_launch():
    run_child("""
        calls = {
            "fathom_calibrate": lambda: L.fathom_calibrate(2, 16, 128, d, d, d, None),
            "fathom_calibrate_klt": lambda: L.fathom_calibrate_klt(2, 16, 128, d, d, d, d, None),
            "fathom_rotate_keys": lambda: L.fathom_rotate_keys(ctypes.byref(s), d, 1, 1, d, d, d, None),
            "fathom_rotate_query": lambda: L.fathom_rotate_query(ctypes.byref(s), d, 1, d, d, None),
            "fathom_quantize_pack": lambda: L.fathom_quantize_pack(ctypes.byref(s), d, 1, d, d, None),
            "fathom_append_block": lambda: L.fathom_append_block(ctypes.byref(s), d, 1, 3, 64, d, d, None),
            "fathom_plan": lambda: L.fathom_plan(ctypes.byref(s), d, d, d, None, d, d, d, None),
            "fathom_plan_fixed": lambda: L.fathom_plan_fixed(ctypes.byref(s), d, d, 32, 4, d, d, None),
            "fathom_gather": lambda: L.fathom_gather(ctypes.byref(s), d, d, d, d, d, 1024, 1024, None),
            "fathom_scan_topk": lambda: L.fathom_scan_topk(ctypes.byref(s), d, d, 0, 0, 0, d, d, d, d, None,
                                                           d, big, None),
            "fathom_exact_topk": lambda: L.fathom_exact_topk(ctypes.byref(s), d, d, d, d, None, d, big, None),
            "fathom_sparse_attn": lambda: L.fathom_sparse_attn(ctypes.byref(s), d, d, d, d, d, d, big, None),
            "fathom_sparse_attn_planes": lambda: L.fathom_sparse_attn_planes(ctypes.byref(s), d, d, d, d, d, d,
                                                                             d, big, None),
            "fathom_sparse_attn_noalloc": lambda: L.fathom_sparse_attn_noalloc(ctypes.byref(s), d, d, d, d, d,
                                                                               None),
            "fathom_dense_attn": lambda: L.fathom_dense_attn(ctypes.byref(s), d, d, d, d, d, big, None),
            "fathom_klt_online": lambda: L.fathom_klt_online(ctypes.byref(s), d, d, d, d, d, big, None),
            "fathom_rel_err": lambda: L.fathom_rel_err(8, 128, d, d, d, None),
            "fathom_set_overlap": lambda: L.fathom_set_overlap(8, 64, d, d, d, None),
        }
        for name, call in calls.items():
            rc = call()
            assert rc == 2, (name, rc, err())
            assert err() == name + ": injected launch failure (FATHOM_FAULT)", (name, err())
        # argument checks still come first
        assert L.fathom_plan(ctypes.byref(s), None, d, d, None, d, d, d, None) == 1 and err() == "q is NULL"
        # host-only calls are not launches
        budgets = (ctypes.c_int32 * 2)()
        errs = (ctypes.c_double * 4)(1.0, 0.5, 1.0, 0.25)
        assert L.fathom_greedy_budgets(2, 2, errs, 24, 8, 28 - 4, budgets) == 0
        # the binding turns the status into an exception
        try:
            B._call("fathom_plan", ctypes.byref(s), d, d, d, None, d, d, d, None)
            raise AssertionError("no exception")
        except B.FathomError as e:
            assert e.status == 2 and "injected launch failure" in str(e)
        print("ok")
    """, "launch")


def test_named_site_fails_only_that_call():
    run_child("""
        assert L.fathom_plan(ctypes.byref(s), d, d, d, None, d, d, d, None) == 2
        assert err() == "fathom_plan: injected launch failure (FATHOM_FAULT)"
        assert L.fathom_scan_topk(ctypes.byref(s), d, d, 0, 0, 0, d, d, d, d, None, d, big, None) == 2
        assert err() == "fathom_scan_topk: injected launch failure (FATHOM_FAULT)"
        # a name that only shares a prefix with a listed one is not injected: with the
        # workspace check failing first, sparse_attn_noalloc's size check answers instead
        s2 = B.make_shape(2048, 1 << 16, 128, 4, 2048)
        assert L.fathom_sparse_attn_noalloc(ctypes.byref(s2), d, d, d, d, d, None) == 1
        assert "scratch" in err()
        print("ok")
    """, "launch:fathom_plan,launch:fathom_sparse_attn,launch:fathom_scan_topk")


def test_unset_or_unknown_sites_inject_nothing():
    for fault in (None, "", "alloc", "launch:fathom_planx", "launchx"):
        run_child("""
            # argument checks answer as usual, and the host-only call succeeds
            assert L.fathom_plan(ctypes.byref(s), None, d, d, None, d, d, d, None) == 1
            assert err() == "q is NULL"
            budgets = (ctypes.c_int32 * 2)()
            errs = (ctypes.c_double * 4)(1.0, 0.5, 1.0, 0.25)
            assert L.fathom_greedy_budgets(2, 2, errs, 24, 8, 24, budgets) == 0
            # a launching call gets past its fault point: noalloc's own size check answers
            s2 = B.make_shape(2048, 1 << 16, 128, 4, 2048)
            assert L.fathom_sparse_attn_noalloc(ctypes.byref(s2), d, d, d, d, d, None) == 1
            assert "scratch" in err()
            print("ok")
        """, fault)
