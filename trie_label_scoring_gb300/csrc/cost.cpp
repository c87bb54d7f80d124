// Speed-of-light cost model of the three classification methods and the
// method picker ("To Classify, Try a Trie Tree", sec. 4). Host only.
//
// Per method (sec. 4.1 Table 2, sec. 4.2, sec. 4.3):
//   trie_tree    q_tail, a = |P| (evaluated positions), V_out = vocab, 1 request
//   letters      q_tail + 2M + 3, a = 1, V_out = M, 1 request
//   trie_decode  q_tail, a = E[1 + depth of the deciding node], V_out = vocab,
//                b = E[branching nodes on the label's path] requests
// then n_tok = L1 + N (q_pre + q_tail + a), K = ceil(n_tok / C), prompt KV
// tokens read R = L1 + N (q_pre + q_tail) (trie_decode: (b - 1) times that),
// B_attn = B_kv (n_tok + R), and the roofline times of the head, the
// projections and the MLP (max of FLOP / Pi and streamed weight bytes / beta)
// and of attention (B_attn / beta). Labels are equally likely (sec. 4.3).
#include <cmath>
#include <cstdio>
#include <string>

#include "trie.h"

namespace quail {

namespace {

struct Shape {
  double q_tail, a, v_out, requests;
};

// b and the expected decode tokens, walking every label's path from the root.
void decode_expectations(const quail_trie& t, double* b, double* a_dec) {
  double sum_b = 0.0, sum_a = 0.0;
  std::vector<int32_t> path;
  for (int32_t m = 0; m < t.num_labels; ++m) {
    path.clear();
    for (int32_t u = t.label_end_node[m]; u >= 0; u = t.parent[u]) path.push_back(u);
    int branching = 0, decide_depth = 0;
    // path is end .. root; step from the root towards the end, stopping at the
    // first node whose subtree holds this label alone (the label is decided)
    for (size_t i = path.size(); i-- > 1;) {
      const int32_t u = path[i];
      if (t.subtree_labels[u] <= 1) break;
      if (t.is_branching[u]) {
        ++branching;
        decide_depth = t.depth[u];
      }
    }
    sum_b += branching;
    sum_a += 1.0 + decide_depth;
  }
  *b = t.num_labels > 0 ? sum_b / t.num_labels : 0.0;
  *a_dec = t.num_labels > 0 ? sum_a / t.num_labels : 0.0;
}

void estimate(const quail_cost_model& md, const quail_cost_workload& w, const Shape& sh, quail_method_cost* c) {
  const double N = w.num_docs;
  c->runnable = 1;
  c->q_tail = sh.q_tail;
  c->a = sh.a;
  c->v_out = sh.v_out;
  c->requests = sh.requests;
  c->n_tok = w.doc_tokens + N * (w.q_pre + sh.q_tail + sh.a);
  c->passes = std::ceil(c->n_tok / w.max_pass_tokens);
  const double prompt = w.doc_tokens + N * (w.q_pre + sh.q_tail);
  c->kv_read_tokens = sh.requests <= 1.0 ? prompt : (sh.requests - 1.0) * prompt;
  c->attn_bytes = md.kv_bytes_per_token * (c->n_tok + c->kv_read_tokens);
  c->head_flops = 2.0 * md.d_model * sh.v_out * N * sh.a;
  c->head_bytes = 2.0 * md.d_model * sh.v_out * c->passes;
  c->t_head = std::fmax(c->head_flops / md.peak_flops, c->head_bytes / md.hbm_bytes_per_s);
  c->t_proj = std::fmax(2.0 * md.proj_params * c->n_tok / md.peak_flops,
                        2.0 * md.proj_params * c->passes / md.hbm_bytes_per_s);
  c->t_mlp = std::fmax(2.0 * md.mlp_params * c->n_tok / md.peak_flops,
                       2.0 * md.mlp_params * c->passes / md.hbm_bytes_per_s);
  c->t_attn = c->attn_bytes / md.hbm_bytes_per_s;
  c->t_classify = c->t_proj + c->t_attn + c->t_mlp + c->t_head;
}

}  // namespace

quail_status estimate_methods_host(const quail_cost_model* md, const quail_cost_workload* w, const quail_trie* t,
                                   quail_method_cost* costs, int32_t* best, std::string* msg) {
  if (md == nullptr || w == nullptr || t == nullptr || costs == nullptr || best == nullptr) {
    *msg = "null argument";
    return QUAIL_ERR_INVALID_ARG;
  }
  if (md->d_model < 1 || md->vocab < 1 || !(md->peak_flops > 0.0) || !(md->hbm_bytes_per_s > 0.0) ||
      !(md->proj_params >= 0.0) || !(md->mlp_params >= 0.0) || !(md->kv_bytes_per_token >= 0.0)) {
    *msg = "cost model: d_model, vocab, peaks must be positive and parameter counts non-negative";
    return QUAIL_ERR_INVALID_ARG;
  }
  if (w->num_docs < 0 || !(w->doc_tokens >= 0.0) || w->q_pre < 0 || w->q_tail < 0 || w->max_pass_tokens < 1) {
    *msg = "cost workload: counts must be non-negative and max_pass_tokens >= 1";
    return QUAIL_ERR_INVALID_ARG;
  }
  double b = 0.0, a_dec = 0.0;
  decode_expectations(*t, &b, &a_dec);
  const Shape shapes[QUAIL_NUM_METHODS] = {
      {static_cast<double>(w->q_tail), a_dec, static_cast<double>(md->vocab), b},         // trie_decode
      {static_cast<double>(w->q_tail), static_cast<double>(t->n_eval()), static_cast<double>(md->vocab), 1.0},
      {static_cast<double>(w->q_tail) + 2.0 * t->num_labels + 3.0, 1.0, static_cast<double>(t->num_labels), 1.0},
  };
  *best = -1;
  for (int i = 0; i < QUAIL_NUM_METHODS; ++i) {
    costs[i] = quail_method_cost{};
    const bool runnable = !(i == QUAIL_METHOD_TRIE_DECODE && (w->need_probabilities || t->has_prefix_labels));
    if (!runnable) continue;
    estimate(*md, *w, shapes[i], &costs[i]);
    if (*best < 0 || costs[i].t_classify < costs[*best].t_classify) *best = i;
  }
  return QUAIL_OK;
}

}  // namespace quail
