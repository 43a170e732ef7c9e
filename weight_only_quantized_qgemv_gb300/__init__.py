"""Weight-only group-quantized GEMV and routed-expert MLP for GB300 (sm_103a).

The computation lives in a CUDA shared library with a C ABI (include/qgemv.h);
this package holds its sources (csrc/), the build step, a thin ctypes binding
with the same entry-point names, and the seeded synthetic workloads.
"""
from ._lib import (QACT_SWIGLU, QACT_SWIGLU_CLAMPED, QFMT_INT3_G64, QFMT_INT4_G, QFMT_INT4_ROW,  # noqa: F401
                   QFMT_INT8_G, QFMT_INT8_ROW, QFMT_MXFP4_E8M0, QFMT_MXFP4_G32, QROUTE_SIGMOID_BIAS, QROUTE_SOFTMAX,
                   QStatusError, library_path, qdequant, qexpert_group, qexpert_group_act, qexpert_group_routed,
                   qexpert_group_launches, qexpert_group_workspace, qgate_up, qgate_up_act, qgemm, qgemm_workspace,
                   qgemv, qroute, qstatus_string)
from ._build import build  # noqa: F401
