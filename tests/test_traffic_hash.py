"""The DRAM-traffic figures bench.py reports are keyed to a hash of the CUDA
sources a kernel is built from (bench.KERNEL_SOURCES); a figure whose hash no
longer matches is reported as null.  That only holds if the hash covers every
header of the kernels' directory that the kernel's file includes, directly or
through another header: checked here, on the sources, without a GPU.  (The
public header include/moe.h, reached from moe_internal.cuh, holds the API's
declarations and constants, no kernel code, and is left out of the hash.)"""
import importlib.util
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "quantized_moe_expert_04_b300", "csrc")


def _bench():
    spec = importlib.util.spec_from_file_location("bench_for_hash", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _local_includes(name, seen=None):
    """Every header of this directory that `name` includes, transitively."""
    seen = set() if seen is None else seen
    with open(os.path.join(CSRC, name), encoding="utf-8") as fh:
        for inc in re.findall(r'^\s*#include\s+"([^"/]+)"', fh.read(), flags=re.M):
            if inc not in seen and os.path.exists(os.path.join(CSRC, inc)):
                seen.add(inc)
                _local_includes(inc, seen)
    return seen


def test_every_included_header_is_hashed():
    bench = _bench()
    for kernel, files in bench.KERNEL_SOURCES.items():
        missing = _local_includes(files[0]) - set(files)
        assert not missing, "%s: %s not in its source hash" % (kernel, sorted(missing))


def test_hash_ignores_comments_and_whitespace_only():
    bench = _bench()
    code = 'int a = 1; // note\n/* block */ const char *s = "x // y";\n'
    assert bench._code_only(code) == bench._code_only("int a=1;\nconst char *s=\"x // y\";")
    assert bench._code_only(code) != bench._code_only('int a = 2; const char *s = "x // y";')
