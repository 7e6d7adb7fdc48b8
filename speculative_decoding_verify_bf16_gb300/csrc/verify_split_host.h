// verify_split_host.h -- what spec_verify.cu needs of the work-list verify
// kernel (verify_split.cu).  Host code only.
#pragma once

#include <cstdint>

#include "spec_verify.h"

namespace split_host {

struct SplitShapeIn {
  int lanes, rows, V, esize, sms, smem_optin;
};

struct SplitShape {
  int chunk;       // pass-1 elements per item
  int nchunk;      // pass-1 chunks per row
  int nchunk2;     // pass-2 chunks per row
  int slot_bytes;  // ring slot
  int nslots;
  int head_bytes;
  int smem;        // dynamic shared memory per CTA
  int grid;        // CTAs (at most one per SM)
  int threads;
};

// Workspace bytes a launch over (lanes, rows, V, element size) needs.
uint64_t workspace_bytes(int lanes, int rows, int V, int esize);

// Rounds the kernel takes: 16-byte aligned rows and at most 2048 lanes.
bool eligible(int lanes, bool aligned);

// The launch shape (SPEC_OK or SPEC_ERR_UNSUPPORTED).
int choose(const SplitShapeIn& in, SplitShape* out);

// Checks the workspace and launches; returns a spec_status.
int launch(const spec_verify_args* a, int dev, int sms, int smem_optin, void* stream);

}  // namespace split_host
