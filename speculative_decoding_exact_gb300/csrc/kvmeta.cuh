// kvmeta.cuh — the metadata-only KV rewind (Muser book Ch. 8 §8.6 item 4:
// the KV checkpoint is a rewind of the length; retained rows stay in place).
#pragma once
#include "common.cuh"
#include "internal.h"

namespace spec {

// seq_len := new_len; pages wholly at or beyond new_len return to the free
// stack, from the highest logical page down.  One thread.
SPEC_DEV void kv_rollback_dev(const KvView& kv, int new_len) {
  const int len = *kv.seq_len;
  const int hi = (len + kv.page_size - 1) / kv.page_size;
  const int lo = (new_len + kv.page_size - 1) / kv.page_size;
  for (int p = hi - 1; p >= lo; --p) {
    const int id = kv.page_table[p];
    if (id >= 0 && *kv.free_top < kv.num_pages) {
      kv.free_stack[*kv.free_top] = id;
      *kv.free_top += 1;
      kv.page_table[p] = -1;
    }
  }
  *kv.seq_len = new_len;
}

}  // namespace spec
