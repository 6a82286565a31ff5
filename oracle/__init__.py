"""fp64 CPU oracle for the Mamba selective scan (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  It compiles ``ssm_oracle.c`` with gcc (no CUDA, no shared code with
the GPU library) and exposes it through ctypes on float64 numpy arrays.
"""

from .oracle import build, scan, step, scan_channels, source_path  # noqa: F401
