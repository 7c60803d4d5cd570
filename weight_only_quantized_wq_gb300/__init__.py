"""GB300-native weight-only quantized matmul: CUDA kernels behind a C ABI
(include/wq.h, libwq.so) and a thin ctypes binding with the same names."""
from .binding import (WQError, wq_check_device, wq_chunk_k, wq_matmul, wq_matmul_ex, wq_pack, wq_packed_bytes,  # noqa: F401
                      wq_matmul_noalloc, wq_matmul_path, wq_status_string, wq_t2_matmul, wq_t2_pack,
                      wq_t2_workspace_bytes, wq_unpack, wq_workspace_bytes)
