"""Host-only test (no GPU) of the per-context address cache that
kla_forward_chunked_noalloc uses for its scratch array: the cache is keyed on
the CUDA context ID, so a new context (after cudaDeviceReset, or one the
caller created) misses and has the address looked up in that context, while
two contexts on one device keep their own entries. The header is compiled
into a small C++ check program with g++."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "bayesian_filtering_linear_gb300", "csrc")


def test_context_address_cache(tmp_path):
    exe = tmp_path / "ctx_cache_check"
    subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(HERE, "host", "ctx_cache_check.cpp"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    assert "FAIL" not in r.stdout and r.stdout.count("ok") == 7, r.stdout
