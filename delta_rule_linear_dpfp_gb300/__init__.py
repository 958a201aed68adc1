"""GB300 (sm_103a) delta-rule fast-weight layer core with the DPFP feature map.

The product is the C-ABI library libfastweight.so (include/fastweight.h),
built in-tree by ``delta_rule_linear_dpfp_gb300.build.build()``.  This package
adds a thin ctypes binding with the same entry-point names
(``delta_rule_linear_dpfp_gb300.binding``) and the seeded synthetic input
generators (``delta_rule_linear_dpfp_gb300.inputs``).
"""
from .binding import (FwError, fw_delta_decode_step, fw_delta_forward,  # noqa: F401
                      fw_delta_forward_workspace_size, fw_device_status, fw_dpfp, fw_linear_forward,
                      fw_linear_forward_workspace_size, fw_delta_backward, fw_delta_backward_workspace_size,
                      fw_delta_forward_projected, fw_delta_forward_projected_workspace_size,
                      fw_decode_stack_step, fw_decode_stack_workspace_size)
