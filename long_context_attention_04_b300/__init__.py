"""B300-native (sm_103a) hybrid compressed attention of DeepSeek-V4: CSA + HCA.

The compute lives in liblca.so (CUDA kernels behind the C ABI of include/lca.h);
`api` is the thin Python binding with the same entry-point names.
"""
from .api import (AttnParams, LcaError, csa_attend, csa_attend_workspace, csa_compress_kv,  # noqa: F401
                  csa_indexer_scores, csa_indexer_topk, csa_indexer_workspace, hca_attend,
                  hca_attend_noalloc, hca_attend_workspace, hca_compress_kv, lca_device_error, lca_gemm_bf16, lca_grouped_oproj,
                  lca_topk, lca_version, lca_window_update, params_from)
