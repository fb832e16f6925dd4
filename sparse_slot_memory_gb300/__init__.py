"""GB300 (sm_103a) forward hot path of the chunked sparse-delta-memory recurrence.

Phase 1 (stable sort of each chunk's write / read slot entries, segmented log-cumsums, flags,
packed positions, sorted rows, A / QK pair triangles) and the Phase-2 decay-and-write run in
hand-written CUDA kernels behind the C ABI of ``include/sdm.h`` (``libsdm_gb300.so``). This
package builds that library in-tree and marshals torch CUDA tensors to it.
"""

from ._build import LIB, build  # noqa: F401
from .api import (  # noqa: F401
    STATS,
    SdmError,
    ShapeSpec,
    alloc_outputs,
    alloc_snapshot,
    alloc_workspace,
    device_status,
    dw,
    dw_saving,
    forward_chunks,
    forward_chunks_saving,
    forward_chunks_noalloc,
    gds,
    gwr,
    pa,
    phase1,
    phase1_saving,
    read,
    workspace_bytes,
)
