"""Build and run the floor measurements (launch, streaming, tensor pipe).

Usage: ``python -m gemms_linear_layers_gb300.floors``.  Compiles
``floors.cu`` for sm_103a next to this file (``_build/floors``) and prints
markdown tables.  The program is stand-alone: it is not part of libtg.so.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)


def main():
    from gemms_linear_layers_gb300 import build
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "floors")
    src = os.path.join(HERE, "floors.cu")
    cmd = [build.nvcc(), *build.ARCH, "-O3", "-std=c++17", f"-I{os.path.join(PKG, 'csrc')}", src, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        return r.returncode
    return subprocess.run([exe]).returncode


if __name__ == "__main__":
    sys.exit(main())
