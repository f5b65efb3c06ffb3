"""CPU oracle for the tree-verify round (test infrastructure only; see
tree_verify.py)."""
