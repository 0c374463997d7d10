"""Off-path arithmetic the source page prints as worked toy examples, kept only to check the
oracle harness (TEST INFRASTRUCTURE; not part of the attention path).

[FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程":
* section "四路残差，算出一个具体输入": four residual streams, new residual =
  post * F(z) + B @ r_old with the worked values z = 6, F(z) = 2z, B = I,
  post = [.25, .5, .75, 1] giving [5, 10, 15, 20]. The page does not print r_old; the test
  states the one r_old consistent with those numbers.
* section "选谁和给多少权重，是两次计算": routed weights are the selected (un-biased) scores
  divided by their sum, times route_scale (1.5 for Flash); the lab prints [0.3, 1.2].
"""
import numpy as np


def mhc_residual_update(r_old, z, F, B, post):
    """new residual streams = post * F(z) + B @ r_old (4 streams)."""
    return np.asarray(post, np.float64) * F(z) + np.asarray(B, np.float64) @ np.asarray(r_old, np.float64)


def routing_weights(scores, bias, k, route_scale):
    """Select the k experts by scores + bias, weight them by the un-biased scores normalised to
    sum to 1, then multiply by route_scale."""
    s = np.asarray(scores, np.float64)
    ids = np.argsort(-(s + np.asarray(bias, np.float64)), kind="stable")[:k]
    w = s[ids] / s[ids].sum()
    return ids, w * route_scale
