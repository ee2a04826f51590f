// stage_event.h -- recording a stage-timing event (moe_set_stage_events) on
// the call's stream.
#pragma once

#include <cuda_runtime.h>

namespace moe {

// Inside a stream capture an external record (a timestamped event node of the
// graph, not a capture-internal dependency); outside one a plain record (the
// runtime refuses the external flag there).
inline cudaError_t record_stage(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    return cudaEventRecordWithFlags(ev, s,
                                    cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

}  // namespace moe
