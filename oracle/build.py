"""Compile the CPU oracle (plain C) into a shared library.

Test infrastructure only: the oracle is built so that the test-suite, the
smoke check and the CPU-baseline leg of the benchmark can call it.
"""
import hashlib
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["ep_oracle.c"]
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libep_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-Wall", "-Wextra"]


def _digest():
    h = hashlib.sha256()
    for name in SOURCES + ["ep_oracle.h"]:
        with open(os.path.join(HERE, name), "rb") as f:
            h.update(f.read())
    h.update(" ".join(CFLAGS).encode())
    return h.hexdigest()


def build(force=False):
    """Build the oracle library if its sources changed; return its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp = os.path.join(BUILD_DIR, "stamp")
    digest = _digest()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc"] + CFLAGS + [os.path.join(HERE, s) for s in SOURCES] + ["-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True))
