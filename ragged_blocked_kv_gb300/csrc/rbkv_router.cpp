// Request routing over independent single-GPU replicas.
//
// InfoQ release note on DeepSpeed-FastGen: throughput scales with the number
// of replicas behind a load balancer (16 replicas, 23.7 queries/s).  Every
// replica runs its own composer and cache; the router only decides which
// replica serves a request.  Policy: the replica with the fewest outstanding
// tokens - the prompt tokens not yet prefilled plus the output tokens not yet
// generated of the requests it holds - takes the next request; ties go to the
// replica holding fewer requests, then to the lowest index.  A replica reports
// the tokens each of its requests has consumed after every pass, and the
// request's end.  Host only; no device work and no communication: callers
// move requests and reports between processes themselves.
#include "rbkv.h"

#include <string>
#include <unordered_map>
#include <vector>

namespace rbkv {
rbkv_status set_error(rbkv_status st, const char* msg);
}

struct rbkv_router {
  struct Req {
    int32_t replica;
    int64_t outstanding;
  };
  std::vector<int64_t> load;      // outstanding tokens per replica
  std::vector<int32_t> active;    // requests held per replica
  std::unordered_map<int64_t, Req> reqs;
};

namespace {
rbkv_status bad(const char* msg) { return rbkv::set_error(RBKV_ERR_INVALID, msg); }
}  // namespace

extern "C" {

rbkv_status rbkv_router_create(int32_t num_replicas, rbkv_router** out) {
  if (!out || num_replicas < 1) return bad("num_replicas must be >= 1");
  try {
    rbkv_router* r = new rbkv_router;
    r->load.assign((size_t)num_replicas, 0);
    r->active.assign((size_t)num_replicas, 0);
    *out = r;
  } catch (...) {
    return bad("out of host memory");
  }
  return RBKV_OK;
}

void rbkv_router_destroy(rbkv_router* r) { delete r; }

rbkv_status rbkv_router_assign(rbkv_router* r, int64_t request_id, int32_t prompt_len,
                               int32_t output_len, int32_t* replica) {
  if (!r || !replica) return bad("router or replica is NULL");
  if (prompt_len < 1 || output_len < 1) return bad("prompt_len and output_len must be >= 1");
  if (r->reqs.count(request_id)) return bad("request id already routed");
  int32_t best = 0;
  for (int32_t i = 1; i < (int32_t)r->load.size(); ++i) {
    if (r->load[i] < r->load[best] ||
        (r->load[i] == r->load[best] && r->active[i] < r->active[best]))
      best = i;
  }
  const int64_t tokens = (int64_t)prompt_len + output_len;
  try {
    r->reqs.emplace(request_id, rbkv_router::Req{best, tokens});
  } catch (...) {
    return bad("out of host memory");
  }
  r->load[best] += tokens;
  r->active[best] += 1;
  *replica = best;
  return RBKV_OK;
}

rbkv_status rbkv_router_progress(rbkv_router* r, int64_t request_id, int32_t tokens) {
  if (!r) return bad("router is NULL");
  auto it = r->reqs.find(request_id);
  if (it == r->reqs.end()) return bad("unknown request id");
  if (tokens < 0 || tokens > it->second.outstanding)
    return bad("tokens must be in [0, the request's outstanding tokens]");
  it->second.outstanding -= tokens;
  r->load[it->second.replica] -= tokens;
  return RBKV_OK;
}

rbkv_status rbkv_router_finish(rbkv_router* r, int64_t request_id) {
  if (!r) return bad("router is NULL");
  auto it = r->reqs.find(request_id);
  if (it == r->reqs.end()) return bad("unknown request id");
  r->load[it->second.replica] -= it->second.outstanding;
  r->active[it->second.replica] -= 1;
  r->reqs.erase(it);
  return RBKV_OK;
}

int64_t rbkv_router_load(const rbkv_router* r, int32_t replica) {
  if (!r || replica < 0 || replica >= (int32_t)r->load.size()) return -1;
  return r->load[replica];
}

int32_t rbkv_router_active(const rbkv_router* r, int32_t replica) {
  if (!r || replica < 0 || replica >= (int32_t)r->active.size()) return -1;
  return r->active[replica];
}

}  // extern "C"
