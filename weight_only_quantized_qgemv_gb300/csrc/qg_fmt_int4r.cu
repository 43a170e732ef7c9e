// Streaming kernels and launchers for int4 codes with one scale per row.
#include "qg_device.cuh"
#define QG_FMT ::qg::FMT_INT4_ROW
#define QG_NAME int4r
#include "qg_fmt_impl.cuh"
