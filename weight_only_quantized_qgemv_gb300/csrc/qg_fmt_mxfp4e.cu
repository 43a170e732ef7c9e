// Streaming kernels and launchers for MXFP4 with ue8m0 scale bytes.
#include "qg_device.cuh"
#define QG_FMT ::qg::FMT_MXFP4_E8M0
#define QG_NAME mxfp4e
#include "qg_fmt_impl.cuh"
