"""Compile the C oracle into oracle/_build/libw4a8_oracle.so with gcc.

Test infrastructure: the product path never loads this library.  The flags
keep every fp32 operation a single IEEE operation in source order
(-ffp-contract=off stops gcc from fusing a*b+c on aarch64 hosts).
"""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "w4a8_oracle.c")
HDR = os.path.join(HERE, "w4a8_oracle.h")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libw4a8_oracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build_oracle(force: bool = False) -> str:
    """Build the oracle shared library if missing or older than its sources."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR), os.path.getmtime(__file__))
        if os.path.getmtime(LIB) >= newest:
            return LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=OUT_DIR)
    os.close(fd)
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB



def build_variant(source_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle to show that the pins catch it)."""
    import shutil
    d = os.path.dirname(out_path)
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "w4a8_oracle_variant.c")
    shutil.copy(HDR, os.path.join(d, "w4a8_oracle.h"))
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *CFLAGS, "-w", src, "-o", out_path, "-lm"], check=True)
    return out_path


if __name__ == "__main__":
    print(build_oracle(force=True))
