"""Builds the fp64 CPU oracle (``oracle/ds4a_oracle.c``) into a shared library.

Test infrastructure only: the oracle is the checker of the CUDA library, never
part of it.  Plain gcc, no vendor code, builds the same on x86_64 and aarch64.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle_ds4a.so")
SOURCES = [os.path.join(HERE, "ds4a_oracle.c")]


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if missing or older than its source; return the .so path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(s) for s in SOURCES)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest_src:
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
           "-o", tmp, *SOURCES, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_oracle(force=True))
