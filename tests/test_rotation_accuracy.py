"""The rotation accuracy study (tests/rotation_accuracy.py) at a small size:
what the rotation is for, checked on synthetic data with the oracle's
quantiser.  Without outliers rotating changes nothing on average; with outlier
channels the unrotated groups containing them lose precision while the rotated
error stays where it was."""
import rotation_accuracy as ra


def test_rotation_keeps_quantisation_error_flat_under_outliers():
    rows = {r["factor"]: r for r in ra.study(n_tokens=256, factors=(1, 16), n_q=8)}
    rot1, rot16 = rows[1]["rotated"], rows[16]["rotated"]
    plain1, plain16 = rows[1]["plain"], rows[16]["plain"]
    # Gaussian vectors: rotation is statistics-preserving
    assert abs(rot1["k_rel_mse"] - plain1["k_rel_mse"]) < 0.1 * plain1["k_rel_mse"]
    # outliers x16: rotated error unchanged, unrotated error roughly doubles
    assert abs(rot16["k_rel_mse"] - rot1["k_rel_mse"]) < 0.15 * rot1["k_rel_mse"]
    assert rot16["k_rel_mse"] < 0.7 * plain16["k_rel_mse"]
    # and the attention output follows
    assert rot16["attn_rel_l2"] < plain16["attn_rel_l2"]
