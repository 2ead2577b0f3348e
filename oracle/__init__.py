"""Oracle for the complex SSD forward and its gradients (test infrastructure only).

Only the tests, the package smoke check and the bench's CPU-baseline leg may
import this package. The product path never does.
"""
from .ssd_oracle import (build, head_mix, naive_grad, naive_grad_inputs, naive_scan,  # noqa: F401
                         naive_scan_inputs, oracle_library_path)
