"""Host-side fault injection (PROJ_FAULT=alloc|encode|launch).

Each failure is made on the host, before anything reaches the device: an
allocation of the library that reports out-of-memory, a tensor-map encoding
that reports failure, a kernel launch refused before it is queued.  The tests
check that every entry point turns it into its status code, that nothing is
leaked (device memory is back to where it was once the handles are
destroyed), and that the process's CUDA context stays usable.  The hook is
read once per process, so each case runs in a child process of its own.

They need the CUDA runtime to reach the failing calls (a handle cannot be
created without a device), hence the gpu mark; no GPU fault, trap or hang is
involved.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

CHILD = r"""
import ctypes, json
import torch
import dense_linear_projection_gb300 as dlp

M, N, K = 16, 2048, 1024
X = torch.randn((M, K), device="cuda").to(torch.bfloat16)
W = (torch.randn((N, K), device="cuda") * 0.03).to(torch.bfloat16)
Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
Xh = X.cpu().pin_memory()
Yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
L = dlp.lib()


def scenario():
    out = {}
    # proj_create, many times: every failed create must release what it took.
    h = None
    for _ in range(20):
        hv = ctypes.c_void_p()
        out["create"] = L.proj_create(ctypes.byref(hv), M, N, K, 0, 0, 0, 0, 0, 0, None)
        if out["create"] == 0:
            h = hv.value
            break
        assert hv.value is None, "a failed proj_create must leave *out NULL"
    if h is not None:
        out["run"] = L.proj_run(h, X.data_ptr(), W.data_ptr(), None, Y.data_ptr(), None)
        out["run_again"] = L.proj_run(h, X.data_ptr(), W.data_ptr(), None, Y.data_ptr(), None)
        n = ctypes.c_size_t(0)
        L.proj_packed_weight_bytes(h, ctypes.byref(n))
        P = torch.empty(n.value // 2, dtype=torch.bfloat16, device="cuda")
        out["pack"] = L.proj_pack_weights(h, W.data_ptr(), P.data_ptr(), None)
        out["run_host"] = L.proj_run_host(h, Xh.data_ptr(), W.data_ptr(), None, Yh.data_ptr(), None)
        out["status"] = L.proj_device_status(h, None)
        out["destroy"] = L.proj_destroy(h)
        del P
    out["selftest"] = L.proj_selftest_wait_timeout(100000, None)
    out["noalloc"] = L.proj_run_noalloc(M, N, K, 0, 0, X.data_ptr(), W.data_ptr(), None, Y.data_ptr(), None)
    out["noalloc_status"] = L.proj_noalloc_device_status(None)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


first = scenario()  # also loads the library's module and kernels (one-time device memory)
free_a = torch.cuda.mem_get_info()[0]
for _ in range(3):
    again = scenario()
free_b = torch.cuda.mem_get_info()[0]
assert again == first, (first, again)
out = dict(first)
out["leak_bytes"] = free_a - free_b
# The context still works: a plain torch kernel and a copy back.
out["context_ok"] = (torch.ones(1000, device="cuda") * 2).sum().item() == 2000.0
print("RESULT " + json.dumps(out))
"""


def run_child(fault: str) -> dict:
    env = dict(os.environ)
    env.pop("PROJ_FAULT", None)
    if fault:
        env["PROJ_FAULT"] = fault
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    lines = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")]
    assert r.returncode == 0 and lines, f"child failed ({fault}):\n{r.stdout}\n{r.stderr}"
    return json.loads(lines[-1][len("RESULT "):])


@pytest.fixture(scope="module")
def lib_built():
    import dense_linear_projection_gb300 as dlp
    dlp.build()


def test_no_fault_baseline(lib_built):
    import dense_linear_projection_gb300 as dlp
    r = run_child("")
    assert r["create"] == dlp.PROJ_OK
    for k in ("run", "run_again", "pack", "run_host", "status", "destroy", "noalloc", "noalloc_status"):
        assert r[k] == dlp.PROJ_OK, (k, r)
    assert r["selftest"] == dlp.PROJ_ERR_DEVICE_TIMEOUT
    assert r["context_ok"] and r["leak_bytes"] <= 0, r


def test_alloc_fault(lib_built):
    # Every device allocation of the library fails: proj_create reports
    # out-of-memory (twenty times, nothing leaked); the allocation-free path
    # is unaffected.
    import dense_linear_projection_gb300 as dlp
    r = run_child("alloc")
    assert r["create"] == dlp.PROJ_ERR_OUT_OF_MEMORY, r
    assert r["selftest"] == dlp.PROJ_ERR_OUT_OF_MEMORY, r
    assert r["noalloc"] == dlp.PROJ_OK and r["noalloc_status"] == dlp.PROJ_OK, r
    assert r["context_ok"] and r["leak_bytes"] <= 0, r


def test_encode_fault(lib_built):
    # Tensor-map encoding fails: every run reports PROJ_ERR_CUDA (again on the
    # second call: no half-built map is cached), the handle is still
    # destroyed cleanly, nothing leaks.
    import dense_linear_projection_gb300 as dlp
    r = run_child("encode")
    assert r["create"] == dlp.PROJ_OK, r
    assert r["run"] == dlp.PROJ_ERR_CUDA and r["run_again"] == dlp.PROJ_ERR_CUDA, r
    assert r["run_host"] == dlp.PROJ_ERR_CUDA and r["noalloc"] == dlp.PROJ_ERR_CUDA, r
    assert r["pack"] == dlp.PROJ_OK, r  # packing encodes no tensor map
    assert r["status"] == dlp.PROJ_OK and r["destroy"] == dlp.PROJ_OK, r
    assert r["context_ok"] and r["leak_bytes"] <= 0, r


def test_launch_fault(lib_built):
    # Every launch is refused before it is queued: runs, packing, host runs,
    # the allocation-free run and the self-test report PROJ_ERR_CUDA; the
    # device status stays clean (no kernel ran) and nothing leaks.
    import dense_linear_projection_gb300 as dlp
    r = run_child("launch")
    assert r["create"] == dlp.PROJ_OK, r
    for k in ("run", "run_again", "pack", "run_host", "noalloc", "selftest"):
        assert r[k] == dlp.PROJ_ERR_CUDA, (k, r)
    assert r["status"] == dlp.PROJ_OK and r["noalloc_status"] == dlp.PROJ_OK, r
    assert r["destroy"] == dlp.PROJ_OK and r["context_ok"] and r["leak_bytes"] <= 0, r
