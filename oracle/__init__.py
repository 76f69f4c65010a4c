"""CPU oracle (test infrastructure only; never imported by the product path)."""
from .gdn_tree_oracle import (RequestResult, check_tree, commit_request, verify_batch,
                              verify_request)

__all__ = ["RequestResult", "check_tree", "commit_request", "verify_batch", "verify_request"]
