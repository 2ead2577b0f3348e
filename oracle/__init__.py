"""Oracle for the complex SSD forward (test infrastructure only).

Only the tests, the package smoke check and the bench's CPU-baseline leg may
import this package. The product path never does.
"""
from .ssd_oracle import build, naive_scan, naive_scan_inputs, oracle_library_path  # noqa: F401
