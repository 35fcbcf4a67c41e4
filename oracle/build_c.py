"""Build the C oracle (oracle/ragged_attention_ref.c) into oracle/liboracle_c.so
with gcc.  Test infrastructure: only tests load the library."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ragged_attention_ref.c")
LIB = os.path.join(HERE, "liboracle_c.so")


def build() -> str:
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler: the C oracle cannot be built")
    subprocess.run([cc, "-O2", "-std=c99", "-shared", "-fPIC", "-o", LIB, SRC, "-lm"], check=True)
    return LIB


if __name__ == "__main__":
    print(build())
